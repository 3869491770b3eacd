// Host-side launchers shared between the translation units of libcoli_moe.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace coli {

enum { DT_F32 = 0, DT_BF16 = 1, DT_I4G128 = 2, DT_MXFP8 = 3, DT_MXFP4 = 4 };

// Stores msg as the calling thread's coli_last_error() text; returns code.
int record_error(int code, const char* msg);

// 2-D tensor map over a row-major [rows][cols] array (the driver's encoder is
// fetched at run time, so the library does not link libcuda).
cudaError_t encode_tmap_2d(CUtensorMap* m, CUtensorMapDataType dt, int elem_bytes, const void* ptr,
                           uint64_t rows, uint64_t cols, int box_cols, int box_rows,
                           CUtensorMapSwizzle swizzle);

// Per-device status word (first device-side error wins).
int* device_status_ptr();  // nullptr if the symbol address cannot be taken

// ---- router (A1) ------------------------------------------------------------
size_t route_scratch_bytes(int T, int d, int E);
// A NaN logit ranks below every other (as -inf) and latches COLI_EDEVICE, so
// every token still gets k distinct ids in [0, E).
cudaError_t launch_route(const void* x, const void* w_r, const float* b_r, int T, int d, int E,
                         int k, int act, int32_t* topk_idx, float* topk_w, float* gap,
                         void* scratch, cudaStream_t st, int* status, int* n_launches);

// ---- dispatch (A2) ------------------------------------------------------------
size_t permute_scratch_bytes(int T, int k, int E);
cudaError_t launch_permute(const int32_t* topk_idx, const void* x, int T, int d, int E, int k,
                           int act, int32_t* counts, int32_t* offsets, int32_t* row_token,
                           int32_t* assign_row, void* x_perm, void* scratch, cudaStream_t st,
                           int* status, int* n_launches);

// ---- expert FFN (A3) ----------------------------------------------------------
// Weights in the handle's layout: gate/up rows interleaved in blocks of 64
// ([E][2f][d]: rows 128b..128b+63 are gate features 64b.., the next 64 the
// matching up features); down [E][d][f]. int4: bytes with each 32-bit word
// holding the 8 reduction indices 8w..8w+7 as nibbles (even indices in the
// low half-word, odd in the high), scales bf16 [rows][cols/128].
struct FfnWeights {
  int wdt;
  const void* w_gu;
  const __nv_bfloat16* s_gu;  // int4 scales
  const void* w_dn;
  const __nv_bfloat16* s_dn;
  const uint8_t* s_gu_u8;     // MX: E8M0 scale bytes [rows][K/32]
  const uint8_t* s_dn_u8;
  // Residency tier (decode path): per-expert device arrays [E] with the base
  // of each expert's weights / scales (an HBM slot or mapped host memory);
  // nullptr when every expert is resident at w_gu + e * (expert bytes).
  const uint8_t* const* tab_gu;
  const uint8_t* const* tab_dn;
  const uint8_t* const* tab_sgu;
  const uint8_t* const* tab_sdn;
};

// Expert residency tier state (device pointers; host_* point at mapped
// pinned host memory). Byte counts are per expert.
struct ResidencyState {
  float* score;         // [E] routing score
  int32_t* slot_of;     // [E] slot holding expert e, or -1
  int32_t* expert_in;   // [S] expert held by a slot, or -1
  int32_t* copy_list;   // [2 P] (expert, slot) pairs of this update
  int32_t* n_copy;      // [1]
  int32_t* promotions;  // [1] running count
  const uint8_t** tab_gu;
  const uint8_t** tab_dn;
  const uint8_t** tab_sgu;
  const uint8_t** tab_sdn;
  uint8_t *host_gu, *host_dn, *host_sgu, *host_sdn;
  uint8_t *slot_gu, *slot_dn, *slot_sgu, *slot_sdn;
  size_t gu_bytes, dn_bytes, sgu_bytes, sdn_bytes;
};
// After a forward: scores from this forward's counts, up to P promotions of
// top-S experts into slots (tables repointed, weights copied host -> slot).
cudaError_t launch_residency_update(const int32_t* counts, int E, int S, int P,
                                    const ResidencyState& R, int grid, cudaStream_t st);

// Tensor-core decode path: streams the weights of every non-empty expert once.
// steps = reduction steps of one down row (f/32 bf16, f/128 int4)
int dec_down_splits(int n_rows, int E, int d, int steps, int n_warps, int max_splits);
// int4: xsum / hsum = 136 * the per-128-group sums of the activation rows
// (launch_group_sums), nullptr for bf16. Gate/up activations: row_token
// nullptr -> x holds the permuted rows (x_perm); otherwise x is [T][d] and
// row r reads x[row_token[r]] (xsum is then per token too).
cudaError_t launch_dec_gateup(const FfnWeights& w, const __nv_bfloat16* x,
                              const int32_t* row_token, const int32_t* offsets, int E, int d,
                              int f, __nv_bfloat16* H, const float* xsum, int grid,
                              cudaStream_t st);
cudaError_t launch_dec_down(const FfnWeights& w, const __nv_bfloat16* H, const int32_t* offsets,
                            int E, int d, int f, int splits, float* y_part, size_t part_stride,
                            const float* hsum, int grid, cudaStream_t st);
cudaError_t launch_group_sums(const __nv_bfloat16* rows, int n_rows, int K, float* out,
                              cudaStream_t st);
int dec_blocks_per_sm();

// fp32 CUDA-core path (f32 activations and weights).
cudaError_t launch_f32_ffn(const float* w_gu, const float* w_dn, const float* x_perm,
                           const int32_t* offsets, int n_rows, int E, int d, int f, float* H,
                           float* y_perm, cudaStream_t st, int* n_launches);

// Block-scaled (MX) experts, decode path: fp16 activations x16 ([T][d]
// through row_token, or [rows][d]), H16 [rows][f] fp16 written by gate/up.
// Values beyond the fp16 range are saturated and latch COLI_EDEVICE.
int mx_blocks_per_sm(int wdt);
cudaError_t launch_to_f16(const void* x_bf16, size_t n, void* x_f16, cudaStream_t st,
                          int* status);
cudaError_t launch_mx_gateup(const FfnWeights& w, const void* x16, const int32_t* row_token,
                             const int32_t* offsets, int E, int d, int f, void* H16, int grid,
                             cudaStream_t st, int* status);
cudaError_t launch_mx_down(const FfnWeights& w, const void* H16, const int32_t* offsets, int E,
                           int d, int f, int splits, float* y_part, size_t part_stride, int grid,
                           cudaStream_t st, int* status);
cudaError_t launch_repack_mx(const void* src_gate, const void* src_up, const void* src_down,
                             const void* sg, const void* su, const void* sd, int wdt, int E,
                             int d, int f, void* dst_gu, void* dst_sgu, void* dst_dn,
                             void* dst_sdn, cudaStream_t st);

// Prefill path: TMA + tcgen05/TMEM grouped GEMM. bf16 weights: both operands
// in shared memory (CTA pairs); int4 / MX weights: dequantised into tensor
// memory by converter warps (k_ffn_tcq.cu).
struct TcPlan;  // defined in k_ffn_tc.cu
struct QPlan;   // defined in k_ffn_tcq.cu
// Whether a layer of this weight format and shape has a tensor-core plan.
bool tc_supported(int wdt, int d, int f);
bool tcq_supported(int wdt, int d, int f);
// 2-D tensor map [rows][cols] of elem_bytes-wide elements, box box_rows x box_cols.
cudaError_t encode_tmap_2d(CUtensorMap* m, CUtensorMapDataType dt, int elem_bytes, const void* ptr,
                           uint64_t rows, uint64_t cols, int box_cols, int box_rows,
                           CUtensorMapSwizzle swizzle);
// x_perm [max_rows][d] and H [max_rows][f] are the handle's buffers: their
// tensor maps are encoded once here (rows past a forward's last group are
// computed from stale data but never stored).
// wdt DT_BF16: w_gu/w_dn bf16 in the handle layout. DT_I4G128: int4 bytes
// plus bf16 scales s_gu/s_dn (q * s rounded to bf16 per weight). DT_MXFP8 /
// DT_MXFP4: MX bytes in the decode layout plus E8M0 scales (exact in bf16
// within its range); mx_general: the weights hold E4M3 NaN codes or scales
// above 2^15, which take the exact fp32 conversion.
cudaError_t tc_plan_create(TcPlan** plan, int wdt, const void* w_gu, const void* w_dn,
                           const void* s_gu, const void* s_dn, int E, int d, int f, int max_rows,
                           const void* x_perm, const void* H, bool mx_general);
void tc_plan_destroy(TcPlan* plan);
cudaError_t tcq_plan_create(QPlan** plan, int wdt, const void* w_gu, const void* w_dn,
                            const void* s_gu, const void* s_dn, int E, int d, int f,
                            int max_rows, const void* x_perm, const void* H, bool general);
void tcq_plan_destroy(QPlan* plan);
cudaError_t launch_tcq_gateup(QPlan* p, const void* x_perm, bool own_x_perm,
                              const int32_t* offsets, void* H, int n_rows, cudaStream_t st,
                              int* status);
cudaError_t launch_tcq_down(QPlan* p, const int32_t* offsets, void* y_perm, bool bf16_out,
                            int n_rows, cudaStream_t st, int* status);
// Sets *flag (device int) to 1 when MX weights hold E4M3 NaN codes
// (MXFP8) or scale bytes above 142.
cudaError_t launch_mx_scan(const void* w, size_t w_bytes, const void* s, size_t s_bytes, int wdt,
                           int* flag, cudaStream_t st);
// H[rows][f] = silu(x_perm Wg^T) * (x_perm Wu^T) per expert group (bf16).
// own_x_perm: x_perm is the plan's buffer (its map is reused), else a map is
// encoded for this call.
cudaError_t launch_tc_gateup(TcPlan* plan, const void* x_perm, bool own_x_perm,
                             const int32_t* offsets, void* H, int n_rows, cudaStream_t st,
                             int* status);
// y_perm[rows][d] = H Wd^T per expert group, fp32 or (bf16_out) bf16 rounded
// to nearest even; H is the plan's buffer.
cudaError_t launch_tc_down(TcPlan* plan, const void* H, const int32_t* offsets, void* y_perm,
                           bool bf16_out, int n_rows, cudaStream_t st, int* status);

// ---- combine (A4) and helpers ----------------------------------------------------
// Rows outside [0, T*k) are skipped and latch COLI_EDEVICE in *status.
cudaError_t launch_combine(const float* y_part, int splits, size_t part_stride,
                           const int32_t* assign_row, const float* topk_w, int T, int k, int d,
                           int out_dt, void* y, cudaStream_t st, int* status);
// Same merge from bf16 rows y_perm [T*k][d] (the prefill forward's output of
// the down projection).
cudaError_t launch_combine_bf16(const __nv_bfloat16* y_perm, const int32_t* assign_row,
                                const float* topk_w, int T, int k, int d, int out_dt, void* y,
                                cudaStream_t st, int* status);
cudaError_t launch_reduce_splits(const float* y_part, int splits, size_t part_stride,
                                 int n_rows, int d, float* y_perm, cudaStream_t st);
cudaError_t launch_repack(const void* src_gate, const void* src_up, const void* src_down,
                          const void* sg, const void* su, const void* sd, int wdt, int E, int d,
                          int f, void* dst_gu, void* dst_sgu, void* dst_dn, void* dst_sdn,
                          cudaStream_t st);
cudaError_t launch_selftest_wait(int spin_limit, int* status, cudaStream_t st);

}  // namespace coli
