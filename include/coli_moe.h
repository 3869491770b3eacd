/*
 * coli_moe — forward pass of one sparse Mixture-of-Experts layer on one GB300
 * (sm_103a), behind a plain C ABI.
 *
 * The layer (the "four atomic operations" of the Colibri overview page,
 * trdm.cn/news/527833, section 2.1):
 *   1. router:   l = x·W_r^T (+ b), p = softmax(l) over the E experts
 *                (gating formula softmax(x·w_gate + b_gate), wzjinhao.cn
 *                "Colibri 是什么", section 3.2);
 *   2. top-k:    the k largest logits (ties: lower expert index first),
 *                gates renormalised over the k chosen: g_j = p_j / sum p;
 *   3. dispatch: assignments grouped by expert id with a stable counting
 *                sort (discosf.com "Colibri 不是一只蜂鸟", section 4.2);
 *   4. experts:  per non-empty expert a SwiGLU FFN,
 *                y = (silu(x·Wg^T) * (x·Wu^T))·Wd^T, no biases (w1 = gate,
 *                w3 = up, w2 = down: overview page section 3.1); experts
 *                without tokens are never read (wzjinhao.cn section 2.3);
 *   5. combine:  y[t] = sum_j g[t][j] * y_perm[row(t, j)], back in token
 *                order (mhpn.cn "Colibri 一个被低估的…", section 2.3).
 *
 * Conventions for every entry point:
 *   - Pointers are DEVICE pointers unless the name says host. `stream` is a
 *     cudaStream_t passed as void* (NULL = legacy default stream).
 *   - Every matrix is row-major. Weights use the nn.Linear "[out][in]"
 *     layout, reduction index contiguous: W_r [E][d], W_gate/W_up [E][f][d],
 *     W_down [E][d][f]. int4 (COLI_I4G128): signed two's-complement nibbles,
 *     the low nibble holding the even reduction index, [..][cols/2] bytes,
 *     with one bf16 scale per 128 consecutive reduction indices of a row,
 *     [..][cols/128]; w = q * s (group-wise int4: wth2jhl.online Colibri deep
 *     dive, section 7.3).
 *   - Return value: COLI_OK (0) or a negative coli_status, errno style
 *     (mhpn.cn page, section 3.3). A message goes to the caller's `err`
 *     buffer where the call has one (truncated to err_len, NUL-terminated)
 *     and always to the calling thread's coli_last_error().
 *   - Arguments are validated before anything is launched. Problems found
 *     on the device (an expert id out of range, a bounded wait that ran out)
 *     never trap: the kernel skips the access, latches the first error code
 *     in a per-device status word and returns; coli_device_status() reports
 *     it.
 *   - Launches are asynchronous on `stream`; buffers must stay alive until
 *     the stream work completes. No entry point but create, destroy, the
 *     host-buffer forward and the status query synchronises.
 */
#ifndef COLI_MOE_H
#define COLI_MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  COLI_OK = 0,
  COLI_EINVAL = -1,       /* bad argument (null pointer, size, dtype, alignment) */
  COLI_ENOMEM = -2,       /* device allocation failed (create only) */
  COLI_ECUDA = -3,        /* a CUDA runtime/driver call failed */
  COLI_EUNSUPPORTED = -4, /* valid but not implemented combination */
  COLI_EDEVICE = -5,      /* a kernel found bad data (e.g. expert id >= E) */
  COLI_ETIMEOUT = -6      /* a bounded device-side wait ran out */
} coli_status;

/* Expert weight formats beyond f32/bf16:
 *   COLI_I4G128: signed int4 nibbles, bf16 scale per 128 reduction indices;
 *   COLI_MXFP8:  OCP Microscaling E4M3 bytes [..][cols], one E8M0 scale byte
 *                (2^(s-127)) per 32 reduction indices [..][cols/32];
 *   COLI_MXFP4:  OCP Microscaling E2M1 nibbles [..][cols/2] (low nibble = even
 *                index), E8M0 scale bytes [..][cols/32].
 * MX formats are the block-scaled low-precision weights of the model families
 * in the wth2jhl.online deep dive's table (MXFP4, FP8). The decode path runs
 * them with fp16 activations (values beyond the fp16 range are saturated and
 * latch COLI_EDEVICE); the prefill path dequantises each weight exactly to a
 * bf16 tensor-core operand (an E4M3/E2M1 value times a power of two; a
 * product beyond bf16's range rounds to it, NaN codes and scales give NaN). */
typedef enum {
  COLI_F32 = 0,
  COLI_BF16 = 1,
  COLI_I4G128 = 2,
  COLI_MXFP8 = 3,
  COLI_MXFP4 = 4
} coli_dtype;

/* Expert-FFN path. AUTO picks DECODE when the mean number of rows per expert
 * (T*k/E) is at most 64, else PREFILL. DECODE streams each active expert's
 * weights once (tensor-core MMA fed straight from HBM); PREFILL is the
 * TMA + tcgen05/TMEM grouped GEMM. Both give the same routing and the same
 * outputs within rounding. F32 layers always use the CUDA-core path.
 * int4 experts run on both: DECODE applies each group's scale to the exact
 * sum of q*x in fp32 (w = q*s exactly); PREFILL dequantises each weight to a
 * bf16 tensor-core operand, q*s rounded once to nearest even (q*s can need 11
 * significant bits, bf16 holds 8: a relative change of at most 2^-9 per
 * weight). A layer with 4-bit experts (int4, MXFP4) and d_model or d_ff
 * equal to 128 has no PREFILL form and runs DECODE whatever `path` asks; a
 * residency-tier layer runs DECODE (PREFILL is rejected at create). */
typedef enum { COLI_PATH_AUTO = 0, COLI_PATH_DECODE = 1, COLI_PATH_PREFILL = 2 } coli_path;

typedef struct {
  int32_t d_model;         /* d: multiple of 64 (int4: of 128) */
  int32_t d_ff;            /* f: multiple of 64 (int4: of 128) */
  int32_t n_experts;       /* E: 1..256 */
  int32_t top_k;           /* k: 1..min(E, 8) */
  int32_t max_tokens;      /* largest T any forward will see (workspace size) */
  int32_t act_dtype;       /* coli_dtype of x, y and W_r: F32 or BF16 */
  int32_t weight_dtype;    /* F32 (with F32 activations); BF16, I4G128, MXFP8 or MXFP4
                              (with BF16) */
  int32_t has_router_bias; /* 0 or 1 */
  int32_t path;            /* coli_path */
  /* Expert residency tier (0 = every expert resident in HBM). With
   * 0 < expert_slots < n_experts, every expert's weights are kept in pinned
   * host memory (Grace memory on a GB300 node) and expert_slots of them also
   * in HBM; the decode kernels read a resident expert from HBM and stream any
   * other straight from host memory over NVLink-C2C. After each forward the
   * hot set follows the routing history: each expert's score becomes
   * 0.75 * score + rows routed to it, and up to max_promotions experts of the
   * top expert_slots by score that are not resident are copied into the
   * slots of resident experts outside that top set (a bounded look-ahead:
   * the copies serve the next forward; wth2jhl.online deep dive, sections
   * 3.1 and 4.2). Placement never changes results (section 8.1): outputs are
   * bit-identical to a fully resident handle. Decode path only (PREFILL is
   * COLI_EUNSUPPORTED), bf16 / int4 / MX experts. */
  int32_t expert_slots;
  int32_t max_promotions;  /* 0..expert_slots promotions per forward */
} coli_moe_config;

typedef struct {
  const void* w_router;  /* [E][d] act dtype */
  const float* b_router; /* [E] f32, or NULL when has_router_bias == 0 */
  const void* w_gate;    /* [E][f][d]   (int4, MXFP4: [E][f][d/2] bytes; MXFP8: bytes) */
  const void* w_up;      /* [E][f][d]   (as w_gate) */
  const void* w_down;    /* [E][d][f]   (int4, MXFP4: [E][d][f/2] bytes; MXFP8: bytes) */
  const void* s_gate;    /* int4: bf16 [E][f][d/128]; MX: u8 [E][f][d/32]; else NULL */
  const void* s_up;      /* as s_gate */
  const void* s_down;    /* int4: bf16 [E][d][f/128]; MX: u8 [E][d][f/32]; else NULL */
} coli_moe_weights;

typedef struct coli_moe coli_moe;

/* ---- library ---------------------------------------------------------- */
const char* coli_version(void);
const char* coli_status_string(int status);
/* Message of the last failing call made by this thread ("" if none). */
const char* coli_last_error(void);
/* First device-side error latched since the last query on the current
 * device (COLI_OK if none); synchronises `stream`, then clears the word. */
int coli_device_status(void* stream, char* err, size_t err_len);

/* ---- layer handle (lifecycle after wzjinhao.cn section 4.3: load, run,
 * free the run state before the model) ----------------------------------- */

/* Copies and repacks the weights into a handle-owned layout (gate/up rows
 * interleaved in blocks of 64; int4 nibbles reordered for in-register
 * dequantisation) and allocates every workspace buffer a forward of up to
 * max_tokens tokens needs (the memory budget is fixed at load time:
 * wzjinhao.cn section 2.3). Synchronises `stream` before returning, so the
 * caller may free its weight buffers afterwards. On failure *out is NULL and
 * nothing is leaked. */
int coli_moe_create(const coli_moe_config* cfg, const coli_moe_weights* weights, void* stream,
                    coli_moe** out, char* err, size_t err_len);

/* y[T][d] = layer(x[T][d]) in the act dtype, 0 <= T <= max_tokens. x and y
 * must be 16-byte aligned and must not overlap. Allocates nothing and never
 * synchronises the host (zero allocation inside inference: mhpn.cn section
 * 3.2). Calls on one handle must not overlap in time. */
int coli_moe_forward(coli_moe* h, const void* x, int32_t T, void* y, void* stream, char* err,
                     size_t err_len);

/* Same layer with HOST buffers x_host[T][d] and y_host[T][d] (act dtype):
 * copies x in, runs the forward, copies y out and synchronises `stream`
 * before returning. Pinned host memory gives the fastest copies. */
int coli_moe_forward_host(coli_moe* h, const void* x_host, int32_t T, void* y_host, void* stream,
                          char* err, size_t err_len);

/* Synchronises `stream` and reports the first device-side error latched
 * since the last query (COLI_EDEVICE / COLI_ETIMEOUT) or COLI_OK. */
int coli_moe_device_status(coli_moe* h, void* stream, char* err, size_t err_len);

/* Device pointers to the last forward's intermediates (valid until the next
 * forward on this handle): topk_idx [T][k] i32, topk_w [T][k] f32, gap [T]
 * f32 (l_(k) - l_(k+1), +inf when k == E), counts [E], offsets [E+1],
 * row_token [T*k], assign_row [T*k] (all i32). Any output may be NULL. */
int coli_moe_debug_buffers(const coli_moe* h, const int32_t** topk_idx, const float** topk_w,
                           const float** gap, const int32_t** counts, const int32_t** offsets,
                           const int32_t** row_token, const int32_t** assign_row);

/* Copies the last forward's intermediates (as listed above; T is that
 * forward's token count) into caller-owned device buffers, asynchronously on
 * `stream`. Any destination may be NULL. */
int coli_moe_copy_debug(const coli_moe* h, int32_t T, int32_t* topk_idx, float* topk_w,
                        float* gap, int32_t* counts, int32_t* offsets, int32_t* row_token,
                        int32_t* assign_row, void* stream);

/* Residency tier state (synchronises `stream`): slot_of[e] (host array of
 * n_experts) receives the HBM slot holding expert e, or -1 when it is read
 * from host memory; *promotions the number of experts copied into slots since
 * create. Either output may be NULL. COLI_EINVAL on a handle without a tier. */
int coli_moe_residency(const coli_moe* h, int32_t* slot_of, int64_t* promotions, void* stream);

/* Path (coli_path, never AUTO) a forward of T tokens takes on this handle. */
int coli_moe_path_for(const coli_moe* h, int32_t T);

/* Per-stage timing with CUDA events recorded on the forward's stream.
 * Stages: 0 router, 1 dispatch, 2 expert gate/up, 3 expert down, 4 combine.
 * coli_moe_stage_times synchronises on the last recorded event, adds the
 * elapsed milliseconds of every timed forward since the last call into
 * ms[0..n), the number of timed forwards into *n_forwards and the number of
 * kernel launches into *n_launches, then resets the sums. The first
 * coli_moe_set_timing(h, 1) creates every event the timed forwards record
 * (so a timed forward still allocates nothing); call it outside any section
 * that may not allocate. */
int coli_moe_set_timing(coli_moe* h, int enable);
int coli_moe_stage_times(coli_moe* h, float* ms, int n, int32_t* n_forwards, int64_t* n_launches);

/* Frees the handle; all stream work on it must have finished. NULL is a no-op. */
void coli_moe_destroy(coli_moe* h);

/* ---- exposed stages ----------------------------------------------------- */

/* Router + softmax + top-k + renormalisation (overview page sections 2.1 and
 * 3.2; gating formula wzjinhao.cn section 3.2; the router emits only k ids
 * and k scores per token: discosf.com section 2.1).
 * x [T][d], w_router [E][d] (act dtype), b_router [E] f32 or NULL ->
 * topk_idx [T][k] i32 (descending logit, lower index first on ties),
 * topk_w [T][k] f32 (renormalised gates), gap [T] f32 or NULL.
 * Logits are fp32 dot products (+ bias in fp32). A NaN logit ranks below
 * every other (as -inf) and latches COLI_EDEVICE, so each token still gets k
 * distinct ids in [0, E). Needs coli_route_scratch_bytes(T, d, E) bytes of
 * device scratch (0 when E <= 32; scratch may then be NULL). */
size_t coli_route_scratch_bytes(int32_t T, int32_t d, int32_t E);
int coli_route_topk(const void* x, const void* w_router, const float* b_router, int32_t T,
                    int32_t d, int32_t E, int32_t k, int32_t act, int32_t* topk_idx,
                    float* topk_w, float* gap, void* scratch, size_t scratch_bytes,
                    void* stream);

/* Dispatch (discosf.com section 4.2 counting sort; overview section 3.3
 * token-to-expert map and expert offsets): counts [E], offsets [E+1]
 * (exclusive prefix), row_token [T*k], assign_row [T*k] and the gathered
 * rows x_perm [T*k][d] = x[row_token[r]] (x_perm may be NULL: then only the
 * counts, offsets and maps are produced and x is not read). Rows of one
 * expert keep token order, so the result is unique and bit-exact. Ids outside [0, E) are
 * skipped (their assign_row entry is set to -1, and counts and offsets leave
 * them out) and latch COLI_EDEVICE. Needs coli_permute_scratch_bytes(T, k, E)
 * bytes of device scratch (256-byte aligned). */
size_t coli_permute_scratch_bytes(int32_t T, int32_t k, int32_t E);
int coli_permute(const int32_t* topk_idx, const void* x, int32_t T, int32_t d, int32_t E,
                 int32_t k, int32_t act, int32_t* counts, int32_t* offsets, int32_t* row_token,
                 int32_t* assign_row, void* x_perm, void* scratch, size_t scratch_bytes,
                 void* stream);

/* Expert FFN on grouped rows with the handle's weights (overview section 3.3
 * per-expert GEMM; only experts with rows are touched). x_perm [n_rows][d]
 * (act dtype), offsets [E+1] as produced by coli_permute (n_rows ==
 * offsets[E] <= max_tokens * k) -> y_perm [n_rows][d] f32. Uses the
 * handle's workspace: do not overlap with a forward on the same handle. */
int coli_expert_ffn(const coli_moe* h, const void* x_perm, const int32_t* offsets,
                    int32_t n_rows, float* y_perm, void* stream);

/* Combine (overview section 2.1 weighted merge; mhpn.cn section 2.3 copy back
 * in token order): y[t] = sum_{j ascending} topk_w[t][j] *
 * y_perm[assign_row[t*k+j]], summed in fp32, written in `out` dtype
 * (bf16 by round-to-nearest-even). y_perm has T*k rows; an assign_row entry
 * outside [0, T*k) (such as the -1 of an assignment coli_permute skipped)
 * contributes nothing, is never dereferenced, and latches COLI_EDEVICE. */
int coli_combine(const float* y_perm, const int32_t* assign_row, const float* topk_w,
                 int32_t T, int32_t k, int32_t d, int32_t out, void* y, void* stream);

/* Dispatch without caller scratch, for callers that cannot allocate device
 * memory where they call it (a plugin inside a host program that owns the
 * device memory pool, a real-time loop that may not allocate after start-up).
 * The pages have no counterpart: it is an addition of this library.
 * Same inputs, outputs and results as coli_permute, but the scratch table
 * lives in a fixed COLI_PERMUTE_STATIC_SCRATCH_BYTES area inside the library
 * that each GPU loading the library holds until the process exits; the call
 * itself makes no cudaMalloc, cudaFree or other allocating call. Batches whose
 * table would not fit (coli_permute_scratch_bytes(T, k, E) >
 * COLI_PERMUTE_STATIC_SCRATCH_BYTES, i.e. T*k > 131072 at E = 256 or
 * T*k > 524288 at E = 64) are rejected with COLI_EINVAL.
 * Set-up: the first call on a device looks up the area's device address
 * (cudaGetSymbolAddress) with that device current and keeps it for later
 * calls. Under CUDA's lazy module loading that lookup may also load the
 * library's device code onto the GPU, which allocates the device image
 * (including this area). A caller that may not allocate after start-up
 * should therefore make one call per device at start-up, before any stream
 * capture: a call with T = 0 (and valid pointers) is enough. The kept address
 * is invalid after cudaDeviceReset; do not use this entry point afterwards in
 * the same process.
 * All calls share the one area and it keeps the last call's table, so calls
 * whose kernels overlap on a GPU (other streams, other threads) race and must
 * be serialised by the caller. */
#define COLI_PERMUTE_STATIC_SCRATCH_BYTES 65536
int coli_permute_noalloc(const int32_t* topk_idx, const void* x, int32_t T, int32_t d,
                         int32_t E, int32_t k, int32_t act, int32_t* counts, int32_t* offsets,
                         int32_t* row_token, int32_t* assign_row, void* x_perm, void* stream);

/* ---- fault-handling self-test ------------------------------------------ */
/* Launches one block that waits on a shared-memory barrier nothing will ever
 * complete, giving up after spin_limit polls: it latches COLI_ETIMEOUT and
 * returns, leaving the context usable. Tests the bounded-wait machinery. */
int coli_selftest_bounded_wait(int32_t spin_limit, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* COLI_MOE_H */
