"""GB300-native forward pass of one sparse Mixture-of-Experts layer."""
