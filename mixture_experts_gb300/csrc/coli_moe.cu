// C ABI of libcoli_moe: validation, handle lifecycle, workspace, stage order.
//
// Lifecycle after the wzjinhao.cn page (section 4.3: load the model, create
// the run state, evaluate, free state before model) with the memory budget
// fixed at load time (same page, section 2.3); errno-style return codes and
// caller-owned message buffers after the mhpn.cn page (section 3.3); no
// allocation and no host synchronisation inside a forward (section 3.2).
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <mutex>
#include <utility>
#include <vector>

#include "../../include/coli_moe.h"
#include "internal.h"

using namespace coli;

namespace {

thread_local char g_last_error[512] = "";

int fail(char* err, size_t err_len, int code, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_last_error, sizeof g_last_error, fmt, ap);
  va_end(ap);
  if (err != nullptr && err_len > 0) {
    strncpy(err, g_last_error, err_len - 1);
    err[err_len - 1] = '\0';
  }
  return code;
}

int ok(char* err, size_t err_len) {
  if (err != nullptr && err_len > 0) err[0] = '\0';
  return COLI_OK;
}

#define CUDA_TRY(call)                                                                   \
  do {                                                                                   \
    cudaError_t e_ = (call);                                                             \
    if (e_ != cudaSuccess)                                                               \
      return fail(err, err_len, COLI_ECUDA, "%s failed: %s", #call, cudaGetErrorString(e_)); \
  } while (0)

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

size_t act_size(int dt) { return dt == COLI_F32 ? 4 : 2; }

}  // namespace

// Per-device status word: a kernel that finds bad data or gives up a bounded
// wait latches its code here (first error wins); read and cleared on query.
static __device__ int g_device_status;

namespace coli {
int record_error(int code, const char* msg) { return fail(nullptr, 0, code, "%s", msg); }

int* device_status_ptr() {
  static std::mutex mu;
  static int* ptrs[128] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (ptrs[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_device_status) == cudaSuccess) ptrs[dev] = static_cast<int*>(p);
  }
  return ptrs[dev];
}
}  // namespace coli

namespace {

constexpr int kStages = 5;
constexpr int kTimingRing = 256;
constexpr int kSplitRows = 8192;  // rows x slices the split-reduction buffer holds
constexpr int kMaxSplits = 32;

struct TimingSet {
  cudaEvent_t ev[kStages + 1] = {};
  bool pending;
  int launches;
};

int read_and_clear_status(cudaStream_t st, char* err, size_t err_len) {
  CUDA_TRY(cudaStreamSynchronize(st));
  int v = 0;
  CUDA_TRY(cudaMemcpyFromSymbol(&v, g_device_status, sizeof v));
  const int zero = 0;
  CUDA_TRY(cudaMemcpyToSymbol(g_device_status, &zero, sizeof zero));
  if (v == COLI_EDEVICE)
    return fail(err, err_len, COLI_EDEVICE, "a kernel found an out-of-range expert id or row");
  if (v == COLI_ETIMEOUT)
    return fail(err, err_len, COLI_ETIMEOUT, "a bounded device-side wait ran out");
  if (v != 0) return fail(err, err_len, COLI_EDEVICE, "device status %d", v);
  return ok(err, err_len);
}

}  // namespace

struct coli_moe {
  coli_moe_config cfg{};
  int device = 0;
  int num_sms = 0;
  int dec_grid = 0;
  std::vector<void*> allocs;
  // weights
  void* w_router = nullptr;
  float* b_router = nullptr;
  FfnWeights w{};
  TcPlan* tc = nullptr;
  // workspace
  int32_t* topk_idx = nullptr;
  float* topk_w = nullptr;
  float* gap = nullptr;
  int32_t* counts = nullptr;
  int32_t* offsets = nullptr;
  int32_t* row_token = nullptr;
  int32_t* assign_row = nullptr;
  void* x_perm = nullptr;
  void* H = nullptr;
  void* y_perm = nullptr;  // fp32, or bf16 on the prefill forward
  float* y_part = nullptr;
  void* route_scratch = nullptr;
  void* perm_scratch = nullptr;
  void* x_stage = nullptr;
  void* y_stage = nullptr;
  float* xsum = nullptr;  // int4: 136 * group sums of the gate/up activations, then of H
  // residency tier (expert_slots > 0)
  bool tier = false;
  ResidencyState rs{};
  std::vector<void*> host_allocs;  // pinned host memory, freed at destroy
  // timing
  bool timing = false;
  TimingSet ring[kTimingRing];
  int ring_next = 0;
  bool ring_init = false;
  double stage_ms[kStages] = {};
  int timed_forwards = 0;
  int64_t launches = 0;

  cudaError_t alloc(void** p, size_t bytes) {
    *p = nullptr;
    if (bytes == 0) return cudaSuccess;
    cudaError_t e = cudaMalloc(p, bytes);
    if (e == cudaSuccess) allocs.push_back(*p);
    return e;
  }
  cudaError_t alloc_host(void** host, uint8_t** dev, size_t bytes) {
    *host = nullptr;
    *dev = nullptr;
    if (bytes == 0) return cudaSuccess;
    cudaError_t e = cudaHostAlloc(host, bytes, cudaHostAllocMapped);
    if (e != cudaSuccess) return e;
    host_allocs.push_back(*host);
    void* d = nullptr;
    e = cudaHostGetDevicePointer(&d, *host, 0);
    *dev = static_cast<uint8_t*>(d);
    return e;
  }
  ~coli_moe() {
    if (tc) tc_plan_destroy(tc);
    for (void* p : allocs) cudaFree(p);
    for (void* p : host_allocs) cudaFreeHost(p);
    for (auto& s : ring)
      for (auto& e : s.ev)
        if (e != nullptr) cudaEventDestroy(e);
  }
};

namespace {

int validate_cfg(const coli_moe_config* c, char* err, size_t err_len) {
  if (c == nullptr) return fail(err, err_len, COLI_EINVAL, "config is NULL");
  if (c->d_model <= 0 || c->d_model % 64)
    return fail(err, err_len, COLI_EINVAL, "d_model=%d must be a positive multiple of 64",
                c->d_model);
  if (c->d_ff <= 0 || c->d_ff % 64)
    return fail(err, err_len, COLI_EINVAL, "d_ff=%d must be a positive multiple of 64", c->d_ff);
  if (c->n_experts < 1 || c->n_experts > 256)
    return fail(err, err_len, COLI_EINVAL, "n_experts=%d must be in [1, 256]", c->n_experts);
  if (c->top_k < 1 || c->top_k > c->n_experts || c->top_k > 8)
    return fail(err, err_len, COLI_EINVAL, "top_k=%d must be in [1, min(E, 8)]", c->top_k);
  if (c->max_tokens < 1 || static_cast<long>(c->max_tokens) * c->top_k > (1L << 24))
    return fail(err, err_len, COLI_EINVAL, "max_tokens=%d out of range", c->max_tokens);
  if (c->act_dtype != COLI_F32 && c->act_dtype != COLI_BF16)
    return fail(err, err_len, COLI_EINVAL, "act_dtype must be F32 or BF16");
  if (c->act_dtype == COLI_F32 && c->weight_dtype != COLI_F32)
    return fail(err, err_len, COLI_EINVAL, "F32 activations need F32 expert weights");
  if (c->act_dtype == COLI_BF16 && c->weight_dtype != COLI_BF16 &&
      c->weight_dtype != COLI_I4G128 && c->weight_dtype != COLI_MXFP8 &&
      c->weight_dtype != COLI_MXFP4)
    return fail(err, err_len, COLI_EINVAL,
                "BF16 activations need BF16, I4G128, MXFP8 or MXFP4 weights");
  if (c->weight_dtype == COLI_I4G128 && (c->d_model % 128 || c->d_ff % 128))
    return fail(err, err_len, COLI_EINVAL, "int4 groups need d_model and d_ff multiples of 128");
  if ((c->weight_dtype == COLI_MXFP8 || c->weight_dtype == COLI_MXFP4) &&
      (c->d_model % 128 || c->d_ff % 128))
    return fail(err, err_len, COLI_EINVAL, "MX weights need d_model and d_ff multiples of 128");
  if (c->path < COLI_PATH_AUTO || c->path > COLI_PATH_PREFILL)
    return fail(err, err_len, COLI_EINVAL, "unknown path %d", c->path);
  if (c->expert_slots < 0 || c->expert_slots > c->n_experts)
    return fail(err, err_len, COLI_EINVAL, "expert_slots=%d outside [0, n_experts]",
                c->expert_slots);
  if (c->expert_slots > 0 && c->expert_slots < c->n_experts) {
    if (c->max_promotions < 0 || c->max_promotions > c->expert_slots)
      return fail(err, err_len, COLI_EINVAL, "max_promotions=%d outside [0, expert_slots]",
                  c->max_promotions);
    if (c->weight_dtype == COLI_F32)
      return fail(err, err_len, COLI_EUNSUPPORTED,
                  "the residency tier serves bf16, int4 and MX experts");
    if (c->path == COLI_PATH_PREFILL)
      return fail(err, err_len, COLI_EUNSUPPORTED,
                  "the residency tier runs on the decode path only");
  }
  return COLI_OK;
}

int pick_path(const coli_moe* h, int T) {
  const auto& c = h->cfg;
  if (c.weight_dtype == COLI_F32) return COLI_PATH_DECODE;  // CUDA-core fp32 path
  if (h->tier || h->tc == nullptr) return COLI_PATH_DECODE;
  if (c.path != COLI_PATH_AUTO) return c.path;
  return static_cast<long>(T) * c.top_k <= 64L * c.n_experts ? COLI_PATH_DECODE
                                                             : COLI_PATH_PREFILL;
}

void timing_mark(coli_moe* h, TimingSet* ts, int i, cudaStream_t st) {
  if (ts) cudaEventRecord(ts->ev[i], st);
}

void harvest(coli_moe* h, TimingSet& ts) {
  if (!ts.pending) return;
  cudaEventSynchronize(ts.ev[kStages]);
  for (int i = 0; i < kStages; ++i) {
    float ms = 0.f;
    if (cudaEventElapsedTime(&ms, ts.ev[i], ts.ev[i + 1]) == cudaSuccess) h->stage_ms[i] += ms;
  }
  h->timed_forwards += 1;
  h->launches += ts.launches;
  ts.pending = false;
}

// Expert FFN over grouped rows (x_perm, offsets) -> y (f32). With row_token
// set (decode path, bf16/int4 experts) the gate/up kernel reads row r's
// activations from x_tok[row_token[r]] and x_perm is not used. When the
// decode path splits the down projection, partial slices go to h->y_part and
// *splits_out > 1 (the caller sums them: the combine directly, the FFN stage
// through a reduction). With allow_bf16 the prefill path writes y_perm as
// bf16 (half the bytes for the combine to read) and sets *y_bf16.
int run_ffn(coli_moe* h, const void* x_perm, const int32_t* offsets, int n_rows, void* y_perm,
            int T, cudaStream_t st, TimingSet* ts, int* launches, int* splits_out, char* err,
            size_t err_len, const void* x_tok = nullptr, const int32_t* row_token = nullptr,
            bool allow_bf16 = false, bool* y_bf16 = nullptr) {
  if (y_bf16) *y_bf16 = false;
  const auto& c = h->cfg;
  const int E = c.n_experts, d = c.d_model, f = c.d_ff;
  int* status = device_status_ptr();
  *splits_out = 1;
  if (c.weight_dtype == COLI_F32) {
    // both projections in one launcher; time them as one stage
    CUDA_TRY(launch_f32_ffn(static_cast<const float*>(h->w.w_gu),
                            static_cast<const float*>(h->w.w_dn),
                            static_cast<const float*>(x_perm), offsets, n_rows, E, d, f,
                            static_cast<float*>(h->H), static_cast<float*>(y_perm), st,
                            launches));
    timing_mark(h, ts, 3, st);
    timing_mark(h, ts, 4, st);
    return COLI_OK;
  }
  const int path = pick_path(h, T);
  if (path == COLI_PATH_PREFILL) {
    // the handle's x_perm has a tensor map made at create; a caller's buffer
    // (the exposed FFN stage) gets one encoded here
    CUDA_TRY(launch_tc_gateup(h->tc, x_perm, x_perm == h->x_perm, offsets, h->H, n_rows, st,
                              status));
    timing_mark(h, ts, 3, st);
    CUDA_TRY(launch_tc_down(h->tc, h->H, offsets, y_perm, allow_bf16, n_rows, st, status));
    if (y_bf16) *y_bf16 = allow_bf16;
    timing_mark(h, ts, 4, st);
    *launches += 2;
    return COLI_OK;
  }
  const int steps_mx = f / 128;
  if (c.weight_dtype == COLI_MXFP8 || c.weight_dtype == COLI_MXFP4) {
    // fp16 activations (token rows, or the caller's permuted rows) in the
    // handle's x_perm buffer, which this path leaves unused otherwise
    const void* xa = row_token ? x_tok : x_perm;
    const int xa_rows = row_token ? T : n_rows;
    CUDA_TRY(launch_to_f16(xa, static_cast<size_t>(xa_rows) * d, h->x_perm, st, status));
    CUDA_TRY(launch_mx_gateup(h->w, h->x_perm, row_token, offsets, E, d, f, h->H, h->dec_grid,
                              st, status));
    timing_mark(h, ts, 3, st);
    int max_splits = kSplitRows / n_rows;
    if (max_splits > kMaxSplits) max_splits = kMaxSplits;
    const int splits = dec_down_splits(n_rows, E, d, steps_mx, h->dec_grid * 8, max_splits);
    if (splits > 1)
      CUDA_TRY(launch_mx_down(h->w, h->H, offsets, E, d, f, splits, h->y_part,
                              static_cast<size_t>(n_rows) * d, h->dec_grid, st, status));
    else
      CUDA_TRY(launch_mx_down(h->w, h->H, offsets, E, d, f, 1, static_cast<float*>(y_perm), 0,
                              h->dec_grid, st, status));
    timing_mark(h, ts, 4, st);
    *launches += 3;
    *splits_out = splits;
    return COLI_OK;
  }
  // gate/up activations: token rows of x through row_token (no x_perm), or
  // the caller's permuted rows
  const bool i4 = c.weight_dtype == COLI_I4G128;
  const void* xa = row_token ? x_tok : x_perm;
  const int xa_rows = row_token ? T : n_rows;
  if (i4) {
    CUDA_TRY(launch_group_sums(static_cast<const __nv_bfloat16*>(xa), xa_rows, d, h->xsum, st));
    *launches += 1;
  }
  CUDA_TRY(launch_dec_gateup(h->w, static_cast<const __nv_bfloat16*>(xa), row_token, offsets, E,
                             d, f, static_cast<__nv_bfloat16*>(h->H), i4 ? h->xsum : nullptr,
                             h->dec_grid, st));
  timing_mark(h, ts, 3, st);
  if (i4) {
    CUDA_TRY(launch_group_sums(static_cast<const __nv_bfloat16*>(h->H), n_rows, f, h->xsum, st));
    *launches += 1;
  }
  const int steps = c.weight_dtype == COLI_I4G128 ? f / 128 : f / 32;
  int max_splits = kSplitRows / n_rows;
  if (max_splits > kMaxSplits) max_splits = kMaxSplits;
  const int splits = dec_down_splits(n_rows, E, d, steps, h->dec_grid * 8, max_splits);
  if (splits > 1) {
    CUDA_TRY(launch_dec_down(h->w, static_cast<const __nv_bfloat16*>(h->H), offsets, E, d, f,
                             splits, h->y_part, static_cast<size_t>(n_rows) * d,
                             i4 ? h->xsum : nullptr, h->dec_grid, st));
  } else {
    CUDA_TRY(launch_dec_down(h->w, static_cast<const __nv_bfloat16*>(h->H), offsets, E, d, f, 1,
                             static_cast<float*>(y_perm), 0, i4 ? h->xsum : nullptr,
                             h->dec_grid, st));
  }
  timing_mark(h, ts, 4, st);
  *launches += 2;
  *splits_out = splits;
  return COLI_OK;
}

}  // namespace

extern "C" {

const char* coli_version(void) { return "coli_moe 0.1 (sm_103a)"; }

const char* coli_status_string(int s) {
  switch (s) {
    case COLI_OK: return "ok";
    case COLI_EINVAL: return "invalid argument";
    case COLI_ENOMEM: return "out of device memory";
    case COLI_ECUDA: return "CUDA error";
    case COLI_EUNSUPPORTED: return "unsupported";
    case COLI_EDEVICE: return "device-side data error";
    case COLI_ETIMEOUT: return "device-side wait timed out";
    default: return "unknown status";
  }
}

const char* coli_last_error(void) { return g_last_error; }

int coli_device_status(void* stream, char* err, size_t err_len) {
  return read_and_clear_status(static_cast<cudaStream_t>(stream), err, err_len);
}

int coli_moe_create(const coli_moe_config* cfg, const coli_moe_weights* wts, void* stream,
                    coli_moe** out, char* err, size_t err_len) {
  if (out == nullptr) return fail(err, err_len, COLI_EINVAL, "out is NULL");
  *out = nullptr;
  int rc = validate_cfg(cfg, err, err_len);
  if (rc) return rc;
  if (wts == nullptr || !wts->w_router || !wts->w_gate || !wts->w_up || !wts->w_down)
    return fail(err, err_len, COLI_EINVAL, "weights and their router/gate/up/down pointers must be set");
  if (cfg->has_router_bias && !wts->b_router)
    return fail(err, err_len, COLI_EINVAL, "has_router_bias=1 but b_router is NULL");
  const bool i4 = cfg->weight_dtype == COLI_I4G128;
  const bool mx = cfg->weight_dtype == COLI_MXFP8 || cfg->weight_dtype == COLI_MXFP4;
  if ((i4 || mx) && (!wts->s_gate || !wts->s_up || !wts->s_down))
    return fail(err, err_len, COLI_EINVAL, "int4 and MX weights need s_gate, s_up and s_down");
  const void* ptrs[] = {wts->w_router, wts->w_gate, wts->w_up, wts->w_down};
  for (const void* p : ptrs)
    if (!aligned16(p)) return fail(err, err_len, COLI_EINVAL, "weight buffers must be 16-byte aligned");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  coli_moe* h = new coli_moe();
  h->cfg = *cfg;
  const int E = cfg->n_experts, d = cfg->d_model, f = cfg->d_ff, k = cfg->top_k;
  const long Tm = cfg->max_tokens, Na = Tm * k;
  const size_t asz = act_size(cfg->act_dtype);
  auto bail = [&](int code, const char* what, cudaError_t e) {
    delete h;
    return fail(err, err_len, code, "%s: %s", what, cudaGetErrorString(e));
  };
  cudaError_t e;
  if ((e = cudaGetDevice(&h->device)) != cudaSuccess) return bail(COLI_ECUDA, "cudaGetDevice", e);
  if ((e = cudaDeviceGetAttribute(&h->num_sms, cudaDevAttrMultiProcessorCount, h->device)) !=
      cudaSuccess)
    return bail(COLI_ECUDA, "device attributes", e);
  h->dec_grid = h->num_sms * (mx ? mx_blocks_per_sm(cfg->weight_dtype) : dec_blocks_per_sm());
  if (device_status_ptr() == nullptr) return bail(COLI_ECUDA, "status word", cudaGetLastError());

  // weights
  const size_t wr_bytes = static_cast<size_t>(E) * d * asz;
  size_t gu_bytes, dn_bytes, sgu_bytes = 0, sdn_bytes = 0;
  if (i4) {
    gu_bytes = static_cast<size_t>(E) * 2 * f * d / 2;
    dn_bytes = static_cast<size_t>(E) * d * f / 2;
    sgu_bytes = static_cast<size_t>(E) * 2 * f * (d / 128) * 2;
    sdn_bytes = static_cast<size_t>(E) * d * (f / 128) * 2;
  } else if (mx) {
    const size_t per = cfg->weight_dtype == COLI_MXFP8 ? 1 : 2;  // elements per byte
    gu_bytes = static_cast<size_t>(E) * 2 * f * d / per;
    dn_bytes = static_cast<size_t>(E) * d * f / per;
    sgu_bytes = static_cast<size_t>(E) * 2 * f * (d / 32);
    sdn_bytes = static_cast<size_t>(E) * d * (f / 32);
  } else {
    const size_t wsz = cfg->weight_dtype == COLI_F32 ? 4 : 2;
    gu_bytes = static_cast<size_t>(E) * 2 * f * d * wsz;
    dn_bytes = static_cast<size_t>(E) * d * f * wsz;
  }
  void *wgu = nullptr, *wdn = nullptr, *sgu = nullptr, *sdn = nullptr;
  const int hsz = cfg->weight_dtype == COLI_F32 ? 4 : 2;
  // residency tier: the expert weights go to pinned host memory instead
  const bool tier = cfg->expert_slots > 0 && cfg->expert_slots < E;
  const int S = tier ? cfg->expert_slots : 0, P = tier ? cfg->max_promotions : 0;
  struct {
    void** p;
    size_t n;
  } plan[] = {
      {&h->w_router, wr_bytes},
      {reinterpret_cast<void**>(&h->b_router), cfg->has_router_bias ? E * sizeof(float) : 0},
      {&wgu, tier ? 0 : gu_bytes},
      {&wdn, tier ? 0 : dn_bytes},
      {&sgu, tier ? 0 : sgu_bytes},
      {&sdn, tier ? 0 : sdn_bytes},
      {reinterpret_cast<void**>(&h->topk_idx), Na * sizeof(int32_t)},
      {reinterpret_cast<void**>(&h->topk_w), Na * sizeof(float)},
      {reinterpret_cast<void**>(&h->gap), Tm * sizeof(float)},
      {reinterpret_cast<void**>(&h->counts), E * sizeof(int32_t)},
      {reinterpret_cast<void**>(&h->offsets), (E + 1) * sizeof(int32_t)},
      {reinterpret_cast<void**>(&h->row_token), Na * sizeof(int32_t)},
      {reinterpret_cast<void**>(&h->assign_row), Na * sizeof(int32_t)},
      {&h->x_perm, Na * d * asz},
      {&h->H, Na * f * static_cast<size_t>(hsz)},
      {reinterpret_cast<void**>(&h->y_perm), Na * d * sizeof(float)},
      {reinterpret_cast<void**>(&h->y_part), static_cast<size_t>(kSplitRows) * d * sizeof(float)},
      {&h->route_scratch, route_scratch_bytes(static_cast<int>(Tm), d, E)},
      {&h->perm_scratch, permute_scratch_bytes(static_cast<int>(Tm), k, E)},
      {&h->x_stage, Tm * d * asz},
      {reinterpret_cast<void**>(&h->xsum),
       i4 ? Na * static_cast<size_t>((d > f ? d : f) / 128) * sizeof(float) : 0},
      {&h->y_stage, Tm * d * asz},
  };
  for (auto& a : plan)
    if ((e = h->alloc(a.p, a.n)) != cudaSuccess) return bail(COLI_ENOMEM, "cudaMalloc", e);
  if (tier) {
    ResidencyState& R = h->rs;
    void* host[4];
    if ((e = h->alloc_host(&host[0], &R.host_gu, gu_bytes)) != cudaSuccess ||
        (e = h->alloc_host(&host[1], &R.host_dn, dn_bytes)) != cudaSuccess ||
        (e = h->alloc_host(&host[2], &R.host_sgu, sgu_bytes)) != cudaSuccess ||
        (e = h->alloc_host(&host[3], &R.host_sdn, sdn_bytes)) != cudaSuccess)
      return bail(COLI_ENOMEM, "pinned host memory for the experts", e);
    wgu = R.host_gu;
    wdn = R.host_dn;
    sgu = R.host_sgu;
    sdn = R.host_sdn;
    R.gu_bytes = gu_bytes / E;
    R.dn_bytes = dn_bytes / E;
    R.sgu_bytes = sgu_bytes / E;
    R.sdn_bytes = sdn_bytes / E;
    struct {
      void** p;
      size_t n;
    } tp[] = {
        {reinterpret_cast<void**>(&R.slot_gu), S * R.gu_bytes},
        {reinterpret_cast<void**>(&R.slot_dn), S * R.dn_bytes},
        {reinterpret_cast<void**>(&R.slot_sgu), S * R.sgu_bytes},
        {reinterpret_cast<void**>(&R.slot_sdn), S * R.sdn_bytes},
        {reinterpret_cast<void**>(&R.tab_gu), E * sizeof(void*)},
        {reinterpret_cast<void**>(&R.tab_dn), E * sizeof(void*)},
        {reinterpret_cast<void**>(&R.tab_sgu), E * sizeof(void*)},
        {reinterpret_cast<void**>(&R.tab_sdn), E * sizeof(void*)},
        {reinterpret_cast<void**>(&R.score), E * sizeof(float)},
        {reinterpret_cast<void**>(&R.slot_of), E * sizeof(int32_t)},
        {reinterpret_cast<void**>(&R.expert_in), S * sizeof(int32_t)},
        {reinterpret_cast<void**>(&R.copy_list), 2 * (P > 0 ? P : 1) * sizeof(int32_t)},
        {reinterpret_cast<void**>(&R.n_copy), sizeof(int32_t)},
        {reinterpret_cast<void**>(&R.promotions), sizeof(int32_t)},
    };
    for (auto& a : tp)
      if ((e = h->alloc(a.p, a.n)) != cudaSuccess) return bail(COLI_ENOMEM, "cudaMalloc", e);
    h->tier = true;
  }
  if ((e = cudaMemcpyAsync(h->w_router, wts->w_router, wr_bytes, cudaMemcpyDefault, st)) !=
      cudaSuccess)
    return bail(COLI_ECUDA, "copy router weights", e);
  if (cfg->has_router_bias &&
      (e = cudaMemcpyAsync(h->b_router, wts->b_router, E * sizeof(float), cudaMemcpyDefault,
                           st)) != cudaSuccess)
    return bail(COLI_ECUDA, "copy router bias", e);
  e = mx ? launch_repack_mx(wts->w_gate, wts->w_up, wts->w_down, wts->s_gate, wts->s_up,
                           wts->s_down, cfg->weight_dtype, E, d, f, wgu, sgu, wdn, sdn, st)
         : launch_repack(wts->w_gate, wts->w_up, wts->w_down, wts->s_gate, wts->s_up,
                         wts->s_down, cfg->weight_dtype, E, d, f, wgu, sgu, wdn, sdn, st);
  if (e != cudaSuccess) return bail(COLI_ECUDA, "repack expert weights", e);
  h->w.wdt = cfg->weight_dtype;
  h->w.w_gu = wgu;
  h->w.w_dn = wdn;
  if (tier) {
    // experts 0..S-1 start in the slots; the tables point every other expert
    // at its host copy
    ResidencyState& R = h->rs;
    const std::pair<uint8_t*, uint8_t*> part[4] = {{R.slot_gu, R.host_gu}, {R.slot_dn, R.host_dn},
                                                   {R.slot_sgu, R.host_sgu}, {R.slot_sdn, R.host_sdn}};
    const size_t per[4] = {R.gu_bytes, R.dn_bytes, R.sgu_bytes, R.sdn_bytes};
    std::vector<const uint8_t*> tab[4];
    for (int i = 0; i < 4; ++i) {
      if (per[i] > 0 &&
          (e = cudaMemcpyAsync(part[i].first, part[i].second, S * per[i], cudaMemcpyDefault,
                               st)) != cudaSuccess)
        return bail(COLI_ECUDA, "initial expert slots", e);
      // expert x < S sits in slot x, the others are read from their host copy
      tab[i].resize(E);
      for (int x = 0; x < E; ++x)
        tab[i][x] = per[i] == 0 ? nullptr
                                : (x < S ? part[i].first : part[i].second) +
                                      static_cast<size_t>(x) * per[i];
    }
    std::vector<int32_t> slot_of(E), expert_in(S);
    for (int x = 0; x < E; ++x) slot_of[x] = x < S ? x : -1;
    for (int x = 0; x < S; ++x) expert_in[x] = x;
    const uint8_t** dst[4] = {R.tab_gu, R.tab_dn, R.tab_sgu, R.tab_sdn};
    for (int i = 0; i < 4; ++i)
      if ((e = cudaMemcpyAsync(dst[i], tab[i].data(), E * sizeof(void*), cudaMemcpyHostToDevice,
                               st)) != cudaSuccess)
        return bail(COLI_ECUDA, "residency tables", e);
    if ((e = cudaMemcpyAsync(R.slot_of, slot_of.data(), E * sizeof(int32_t),
                             cudaMemcpyHostToDevice, st)) != cudaSuccess ||
        (e = cudaMemcpyAsync(R.expert_in, expert_in.data(), S * sizeof(int32_t),
                             cudaMemcpyHostToDevice, st)) != cudaSuccess ||
        (e = cudaMemsetAsync(R.score, 0, E * sizeof(float), st)) != cudaSuccess ||
        (e = cudaMemsetAsync(R.promotions, 0, sizeof(int32_t), st)) != cudaSuccess ||
        (e = cudaMemsetAsync(R.n_copy, 0, sizeof(int32_t), st)) != cudaSuccess ||
        (e = cudaStreamSynchronize(st)) != cudaSuccess)  // the host tables above go out of scope
      return bail(COLI_ECUDA, "residency state", e);
    h->w.tab_gu = R.tab_gu;
    h->w.tab_dn = R.tab_dn;
    h->w.tab_sgu = R.sgu_bytes ? R.tab_sgu : nullptr;
    h->w.tab_sdn = R.sdn_bytes ? R.tab_sdn : nullptr;
  }
  h->w.s_gu_u8 = mx ? static_cast<const uint8_t*>(sgu) : nullptr;
  h->w.s_dn_u8 = mx ? static_cast<const uint8_t*>(sdn) : nullptr;
  h->w.s_gu = static_cast<const __nv_bfloat16*>(sgu);
  h->w.s_dn = static_cast<const __nv_bfloat16*>(sdn);
  if (cfg->weight_dtype != COLI_F32 && !tier && tc_supported(cfg->weight_dtype, d, f)) {
    // MX weights outside the converters' fast range take their exact path
    int general = 0;
    if (mx) {
      int* flag = nullptr;
      if ((e = h->alloc(reinterpret_cast<void**>(&flag), sizeof(int))) != cudaSuccess ||
          (e = cudaMemsetAsync(flag, 0, sizeof(int), st)) != cudaSuccess ||
          (e = launch_mx_scan(wgu, gu_bytes, sgu, sgu_bytes, cfg->weight_dtype, flag, st)) !=
              cudaSuccess ||
          (e = launch_mx_scan(wdn, dn_bytes, sdn, sdn_bytes, cfg->weight_dtype, flag, st)) !=
              cudaSuccess ||
          (e = cudaMemcpyAsync(&general, flag, sizeof(int), cudaMemcpyDeviceToHost, st)) !=
              cudaSuccess ||
          (e = cudaStreamSynchronize(st)) != cudaSuccess)
        return bail(COLI_ECUDA, "MX weight scan", e);
    }
    if ((e = tc_plan_create(&h->tc, cfg->weight_dtype, wgu, wdn, sgu, sdn, E, d, f,
                            static_cast<int>(Na), h->x_perm, h->H, general != 0)) != cudaSuccess)
      return bail(COLI_ECUDA, "tensor-core plan", e);
  }
  if ((e = cudaStreamSynchronize(st)) != cudaSuccess) return bail(COLI_ECUDA, "create sync", e);
  *out = h;
  return ok(err, err_len);
}

int coli_moe_forward(coli_moe* h, const void* x, int32_t T, void* y, void* stream, char* err,
                     size_t err_len) {
  if (h == nullptr) return fail(err, err_len, COLI_EINVAL, "handle is NULL");
  const auto& c = h->cfg;
  if (T < 0 || T > c.max_tokens)
    return fail(err, err_len, COLI_EINVAL, "T=%d outside [0, max_tokens=%d]", T, c.max_tokens);
  if (T == 0) return ok(err, err_len);
  if (x == nullptr || y == nullptr) return fail(err, err_len, COLI_EINVAL, "x and y must be set");
  if (!aligned16(x) || !aligned16(y))
    return fail(err, err_len, COLI_EINVAL, "x and y must be 16-byte aligned");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int E = c.n_experts, d = c.d_model, k = c.top_k, n_rows = T * k;
  int* status = device_status_ptr();
  TimingSet* ts = nullptr;
  if (h->timing && h->ring_init) {  // events were made by coli_moe_set_timing
    ts = &h->ring[h->ring_next];
    h->ring_next = (h->ring_next + 1) % kTimingRing;
    harvest(h, *ts);
    ts->launches = 0;
  }
  int launches = 0;
  timing_mark(h, ts, 0, st);
  CUDA_TRY(launch_route(x, h->w_router, h->b_router, T, d, E, k, c.act_dtype, h->topk_idx,
                        h->topk_w, h->gap, h->route_scratch, st, status, &launches));
  timing_mark(h, ts, 1, st);
  // the decode kernels read token rows of x themselves: no x_perm copy
  const bool gather = c.weight_dtype != COLI_F32 && pick_path(h, T) == COLI_PATH_DECODE;
  CUDA_TRY(launch_permute(h->topk_idx, x, T, d, E, k, c.act_dtype, h->counts, h->offsets,
                          h->row_token, h->assign_row, gather ? nullptr : h->x_perm,
                          h->perm_scratch, st, status, &launches));
  timing_mark(h, ts, 2, st);
  int splits = 1;
  bool y_bf16 = false;
  int rc = run_ffn(h, h->x_perm, h->offsets, n_rows, h->y_perm, T, st, ts, &launches, &splits,
                   err, err_len, gather ? x : nullptr, gather ? h->row_token : nullptr,
                   /*allow_bf16=*/c.act_dtype == COLI_BF16, &y_bf16);
  if (rc) return rc;
  if (y_bf16) {
    CUDA_TRY(launch_combine_bf16(static_cast<const __nv_bfloat16*>(h->y_perm), h->assign_row,
                                 h->topk_w, T, k, d, c.act_dtype, y, st, status));
  } else {
    const float* part = splits > 1 ? h->y_part : static_cast<const float*>(h->y_perm);
    CUDA_TRY(launch_combine(part, splits, static_cast<size_t>(n_rows) * d, h->assign_row,
                            h->topk_w, T, k, d, c.act_dtype, y, st, status));
  }
  launches += 1;
  if (h->tier && c.max_promotions > 0) {
    // the hot set follows this forward's routing; copies serve the next one
    CUDA_TRY(launch_residency_update(h->counts, E, c.expert_slots, c.max_promotions, h->rs,
                                     h->num_sms * 4, st));
    launches += 2;
  }
  timing_mark(h, ts, 5, st);
  if (ts) {
    ts->launches = launches;
    ts->pending = true;
  }
  return ok(err, err_len);
}

int coli_moe_forward_host(coli_moe* h, const void* x_host, int32_t T, void* y_host, void* stream,
                          char* err, size_t err_len) {
  if (h == nullptr) return fail(err, err_len, COLI_EINVAL, "handle is NULL");
  if (T < 0 || T > h->cfg.max_tokens)
    return fail(err, err_len, COLI_EINVAL, "T=%d outside [0, max_tokens=%d]", T,
                h->cfg.max_tokens);
  if (T == 0) return ok(err, err_len);
  if (x_host == nullptr || y_host == nullptr)
    return fail(err, err_len, COLI_EINVAL, "x_host and y_host must be set");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const size_t bytes = static_cast<size_t>(T) * h->cfg.d_model * act_size(h->cfg.act_dtype);
  CUDA_TRY(cudaMemcpyAsync(h->x_stage, x_host, bytes, cudaMemcpyHostToDevice, st));
  int rc = coli_moe_forward(h, h->x_stage, T, h->y_stage, stream, err, err_len);
  if (rc) return rc;
  CUDA_TRY(cudaMemcpyAsync(y_host, h->y_stage, bytes, cudaMemcpyDeviceToHost, st));
  CUDA_TRY(cudaStreamSynchronize(st));
  return ok(err, err_len);
}

int coli_moe_device_status(coli_moe* h, void* stream, char* err, size_t err_len) {
  if (h == nullptr) return fail(err, err_len, COLI_EINVAL, "handle is NULL");
  return read_and_clear_status(static_cast<cudaStream_t>(stream), err, err_len);
}

int coli_moe_debug_buffers(const coli_moe* h, const int32_t** topk_idx, const float** topk_w,
                           const float** gap, const int32_t** counts, const int32_t** offsets,
                           const int32_t** row_token, const int32_t** assign_row) {
  if (h == nullptr) return fail(nullptr, 0, COLI_EINVAL, "handle is NULL");
  if (topk_idx) *topk_idx = h->topk_idx;
  if (topk_w) *topk_w = h->topk_w;
  if (gap) *gap = h->gap;
  if (counts) *counts = h->counts;
  if (offsets) *offsets = h->offsets;
  if (row_token) *row_token = h->row_token;
  if (assign_row) *assign_row = h->assign_row;
  return COLI_OK;
}

int coli_moe_copy_debug(const coli_moe* h, int32_t T, int32_t* topk_idx, float* topk_w,
                        float* gap, int32_t* counts, int32_t* offsets, int32_t* row_token,
                        int32_t* assign_row, void* stream) {
  char* err = nullptr;
  size_t err_len = 0;
  if (h == nullptr) return fail(err, err_len, COLI_EINVAL, "handle is NULL");
  if (T < 0 || T > h->cfg.max_tokens) return fail(err, err_len, COLI_EINVAL, "bad T=%d", T);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const size_t na = static_cast<size_t>(T) * h->cfg.top_k, E = h->cfg.n_experts;
  struct {
    void* dst;
    const void* src;
    size_t n;
  } cp[] = {{topk_idx, h->topk_idx, na * 4}, {topk_w, h->topk_w, na * 4},
            {gap, h->gap, static_cast<size_t>(T) * 4}, {counts, h->counts, E * 4},
            {offsets, h->offsets, (E + 1) * 4}, {row_token, h->row_token, na * 4},
            {assign_row, h->assign_row, na * 4}};
  for (auto& c : cp)
    if (c.dst != nullptr && c.n > 0)
      CUDA_TRY(cudaMemcpyAsync(c.dst, c.src, c.n, cudaMemcpyDeviceToDevice, st));
  return COLI_OK;
}

int coli_moe_residency(const coli_moe* h, int32_t* slot_of, int64_t* promotions, void* stream) {
  char* err = nullptr;
  size_t err_len = 0;
  if (h == nullptr) return fail(err, err_len, COLI_EINVAL, "handle is NULL");
  if (!h->tier) return fail(err, err_len, COLI_EINVAL, "the handle has no residency tier");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  CUDA_TRY(cudaStreamSynchronize(st));
  if (slot_of)
    CUDA_TRY(cudaMemcpy(slot_of, h->rs.slot_of, h->cfg.n_experts * sizeof(int32_t),
                        cudaMemcpyDeviceToHost));
  if (promotions) {
    int32_t p = 0;
    CUDA_TRY(cudaMemcpy(&p, h->rs.promotions, sizeof p, cudaMemcpyDeviceToHost));
    *promotions = p;
  }
  return COLI_OK;
}

int coli_moe_path_for(const coli_moe* h, int32_t T) {
  if (h == nullptr) return fail(nullptr, 0, COLI_EINVAL, "handle is NULL");
  return pick_path(h, T);
}

int coli_moe_set_timing(coli_moe* h, int enable) {
  char* err = nullptr;
  size_t err_len = 0;
  if (h == nullptr) return fail(err, err_len, COLI_EINVAL, "handle is NULL");
  if (enable && !h->ring_init) {
    // every event the timed forwards will record is made here, so a forward
    // never creates one
    for (auto& ts : h->ring) {
      for (auto& ev : ts.ev) {
        const cudaError_t e = cudaEventCreate(&ev);
        if (e != cudaSuccess) {
          ev = nullptr;
          return fail(err, err_len, COLI_ECUDA, "cudaEventCreate: %s", cudaGetErrorString(e));
        }
      }
      ts.pending = false;
    }
    h->ring_init = true;
  }
  h->timing = enable != 0;
  return COLI_OK;
}

int coli_moe_stage_times(coli_moe* h, float* ms, int n, int32_t* n_forwards, int64_t* n_launches) {
  if (h == nullptr) return fail(nullptr, 0, COLI_EINVAL, "handle is NULL");
  if (h->ring_init)
    for (auto& s : h->ring) harvest(h, s);
  for (int i = 0; i < n && i < kStages; ++i) ms[i] = static_cast<float>(h->stage_ms[i]);
  if (n_forwards) *n_forwards = h->timed_forwards;
  if (n_launches) *n_launches = h->launches;
  for (double& v : h->stage_ms) v = 0.0;
  h->timed_forwards = 0;
  h->launches = 0;
  return COLI_OK;
}

void coli_moe_destroy(coli_moe* h) { delete h; }

// ---- stages ---------------------------------------------------------------------------

size_t coli_route_scratch_bytes(int32_t T, int32_t d, int32_t E) {
  if (T <= 0 || d <= 0 || E <= 0) return 0;
  return route_scratch_bytes(T, d, E);
}

int coli_route_topk(const void* x, const void* w_router, const float* b_router, int32_t T,
                    int32_t d, int32_t E, int32_t k, int32_t act, int32_t* topk_idx,
                    float* topk_w, float* gap, void* scratch, size_t scratch_bytes,
                    void* stream) {
  char* err = nullptr;
  size_t err_len = 0;
  if (T < 0 || d <= 0 || d % 64 || E < 1 || E > 256 || k < 1 || k > E || k > 8)
    return fail(err, err_len, COLI_EINVAL, "bad sizes T=%d d=%d E=%d k=%d", T, d, E, k);
  if (act != COLI_F32 && act != COLI_BF16) return fail(err, err_len, COLI_EINVAL, "bad act dtype");
  if (T == 0) return ok(err, err_len);
  if (!x || !w_router || !topk_idx || !topk_w)
    return fail(err, err_len, COLI_EINVAL, "x, w_router, topk_idx and topk_w must be set");
  if (!aligned16(x) || !aligned16(w_router))
    return fail(err, err_len, COLI_EINVAL, "x and w_router must be 16-byte aligned");
  const size_t need = route_scratch_bytes(T, d, E);
  if (need > 0 && (scratch == nullptr || scratch_bytes < need))
    return fail(err, err_len, COLI_EINVAL, "router needs %zu bytes of scratch", need);
  CUDA_TRY(launch_route(x, w_router, b_router, T, d, E, k, act, topk_idx, topk_w, gap, scratch,
                        static_cast<cudaStream_t>(stream), device_status_ptr(), nullptr));
  return COLI_OK;
}

size_t coli_permute_scratch_bytes(int32_t T, int32_t k, int32_t E) {
  if (T <= 0 || k <= 0 || E <= 0) return 0;
  return permute_scratch_bytes(T, k, E);
}

int coli_permute(const int32_t* topk_idx, const void* x, int32_t T, int32_t d, int32_t E,
                 int32_t k, int32_t act, int32_t* counts, int32_t* offsets, int32_t* row_token,
                 int32_t* assign_row, void* x_perm, void* scratch, size_t scratch_bytes,
                 void* stream) {
  char* err = nullptr;
  size_t err_len = 0;
  if (T < 0 || d <= 0 || d % 64 || E < 1 || E > 256 || k < 1 || k > E ||
      static_cast<long>(T) * k > (1L << 24))
    return fail(err, err_len, COLI_EINVAL, "bad sizes T=%d d=%d E=%d k=%d", T, d, E, k);
  if (act != COLI_F32 && act != COLI_BF16) return fail(err, err_len, COLI_EINVAL, "bad act dtype");
  if (!topk_idx || !counts || !offsets || !row_token || !assign_row)
    return fail(err, err_len, COLI_EINVAL, "topk_idx, counts, offsets, row_token, assign_row must be set");
  if (x_perm != nullptr && (x == nullptr || !aligned16(x) || !aligned16(x_perm)))
    return fail(err, err_len, COLI_EINVAL, "x and x_perm must be set and 16-byte aligned");
  const size_t need = permute_scratch_bytes(T, k, E);
  if (need > 0 && (scratch == nullptr || scratch_bytes < need ||
                   (reinterpret_cast<uintptr_t>(scratch) & 255u)))
    return fail(err, err_len, COLI_EINVAL, "permute needs %zu bytes of 256-byte aligned scratch",
                need);
  CUDA_TRY(launch_permute(topk_idx, x, T, d, E, k, act, counts, offsets, row_token, assign_row,
                          x_perm, scratch, static_cast<cudaStream_t>(stream), device_status_ptr(),
                          nullptr));
  return COLI_OK;
}

int coli_expert_ffn(const coli_moe* hc, const void* x_perm, const int32_t* offsets,
                    int32_t n_rows, float* y_perm, void* stream) {
  char* err = nullptr;
  size_t err_len = 0;
  coli_moe* h = const_cast<coli_moe*>(hc);
  if (h == nullptr) return fail(err, err_len, COLI_EINVAL, "handle is NULL");
  if (n_rows < 0 || static_cast<long>(n_rows) > static_cast<long>(h->cfg.max_tokens) * h->cfg.top_k)
    return fail(err, err_len, COLI_EINVAL, "n_rows=%d outside [0, max_tokens*k]", n_rows);
  if (n_rows == 0) return ok(err, err_len);
  if (!x_perm || !offsets || !y_perm)
    return fail(err, err_len, COLI_EINVAL, "x_perm, offsets and y_perm must be set");
  if (!aligned16(x_perm) || !aligned16(y_perm))
    return fail(err, err_len, COLI_EINVAL, "x_perm and y_perm must be 16-byte aligned");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int launches = 0, splits = 1;
  // the path follows the token count the rows came from
  const int T = (n_rows + h->cfg.top_k - 1) / h->cfg.top_k;
  int rc = run_ffn(h, x_perm, offsets, n_rows, y_perm, T, st, nullptr, &launches, &splits, err,
                   err_len);
  if (rc) return rc;
  if (splits > 1)
    CUDA_TRY(launch_reduce_splits(h->y_part, splits, static_cast<size_t>(n_rows) * h->cfg.d_model,
                                  n_rows, h->cfg.d_model, y_perm, st));
  return COLI_OK;
}

int coli_combine(const float* y_perm, const int32_t* assign_row, const float* topk_w, int32_t T,
                 int32_t k, int32_t d, int32_t out, void* y, void* stream) {
  char* err = nullptr;
  size_t err_len = 0;
  if (T < 0 || k < 1 || k > 256 || d <= 0 || d % 4 || static_cast<long>(T) * k > (1L << 30))
    return fail(err, err_len, COLI_EINVAL, "bad sizes T=%d k=%d d=%d", T, k, d);
  if (out != COLI_F32 && out != COLI_BF16) return fail(err, err_len, COLI_EINVAL, "bad out dtype");
  if (T == 0) return ok(err, err_len);
  if (!y_perm || !assign_row || !topk_w || !y)
    return fail(err, err_len, COLI_EINVAL, "y_perm, assign_row, topk_w and y must be set");
  if (!aligned16(y_perm) || (reinterpret_cast<uintptr_t>(y) & (out == COLI_F32 ? 15u : 7u)))
    return fail(err, err_len, COLI_EINVAL, "y_perm must be 16-byte and y 16/8-byte aligned");
  CUDA_TRY(launch_combine(y_perm, 1, 0, assign_row, topk_w, T, k, d, out, y,
                          static_cast<cudaStream_t>(stream), device_status_ptr()));
  return COLI_OK;
}

int coli_selftest_bounded_wait(int32_t spin_limit, void* stream) {
  char* err = nullptr;
  size_t err_len = 0;
  if (spin_limit < 1) return fail(err, err_len, COLI_EINVAL, "spin_limit must be >= 1");
  CUDA_TRY(launch_selftest_wait(spin_limit, device_status_ptr(), static_cast<cudaStream_t>(stream)));
  return COLI_OK;
}

}  // extern "C"
