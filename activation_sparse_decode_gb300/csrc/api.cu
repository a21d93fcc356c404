// C ABI of libsffn: argument validation, workspace layout and the launch
// sequence of the predictor-gated sparse FFN (declared in include/sffn.h).

#include <algorithm>
#include <cstddef>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <numeric>
#include <new>
#include <string>
#include <vector>

#include <cublasLt.h>

#include "../../include/sffn.h"
#include "kernels.cuh"

// cuBLASLt descriptors of the dense fallback's two GEMMs for one batch size.
struct DensePlan {
  bool built = false, ok = false;
  cublasLtMatmulDesc_t op1 = nullptr, op2 = nullptr;
  cublasLtMatrixLayout_t w1 = nullptr, x1 = nullptr, d1 = nullptr, w2 = nullptr, a2 = nullptr, y2 = nullptr;
  cublasLtMatmulAlgo_t algo1{}, algo2{};
};

using namespace sffn;

struct sffn_layer {
  sffn_layer_desc desc;
  int device = 0;
  int sms = 0;
  size_t smem_optin = 0;
  int esize = 0;
  int W = 0;           // mask words per token
  int kc_elems = 0;    // predictor K-chunk
  int KS = 0;          // predictor K-chunks
  int kc32 = 0;        // predictor K-chunk when one block holds up to 32 tokens
  int KS32 = 0;
  int KStok = 0;       // K-chunks of the lane-per-token hidden-layer kernel (17-32 tokens)
  int RG = 0;          // predictor row groups
  int score_grid = 0;  // blocks of the score kernel
  int gather_grid = 0; // blocks of the gather kernel (one per SM)
  int max_bt = 0;      // tokens per gather pass
  GatherConfig gcfg[3];  // tokens per pass 1, 2, 4
  bool gcfg_ok[3] = {false, false, false};
  size_t wstride = 0;    // bytes between consecutive neurons' rows of each weight matrix
  LayerConfig lcfg{};    // single-launch batch-1 layer kernel
  bool lcfg_ok = false;
  int layer_grid = 0;    // its blocks: two per SM when two fit, else one
  int layer_cluster = 0;  // > 1: launched in clusters of this many blocks (every cluster co-resident)
  cublasLtHandle_t lt = nullptr;  // dense fallback (created when the layer enables it)
  DensePlan plans[33];            // per batch size
  bool fused() const { return lcfg_ok && !(desc.flags & SFFN_FLAG_MULTI_KERNEL); }
  bool dense_for(int batch) const { return lt != nullptr && batch >= desc.dense_min_batch; }
  ~sffn_layer() {
    for (auto& p : plans) {
      if (p.op1) cublasLtMatmulDescDestroy(p.op1);
      if (p.op2) cublasLtMatmulDescDestroy(p.op2);
      for (auto l : {p.w1, p.x1, p.d1, p.w2, p.a2, p.y2})
        if (l) cublasLtMatrixLayoutDestroy(l);
    }
    if (lt) cublasLtDestroy(lt);
  }
};

namespace {

thread_local std::string g_err;
constexpr int kMinStages2 = 4;  // ring stages a block needs for the two-blocks-per-SM layer kernel
int64_t g_wait_ns = 1000000000LL;  // 1 s
// Profiling hook: the next g_prof_n dominant-kernel launches are bracketed by
// event pairs g_prof_start[i], g_prof_stop[i], i counting launches from the
// last sffn_set_profile_events call (host-side, at launch or capture time).
std::vector<cudaEvent_t> g_prof_start, g_prof_stop;
size_t g_prof_next = 0;

constexpr int kVersion = 1;

sffn_status fail(sffn_status st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_err = buf;
  return st;
}

sffn_status cuda_fail(cudaError_t e, const char* where) {
  return fail(SFFN_ERR_CUDA, "%s: %s", where, cudaGetErrorString(e));
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

int bt_slot(int bt) { return bt == 1 ? 0 : bt == 2 ? 1 : 2; }

struct WsLayout {
  size_t hdr, flags, tickets, h_part, h, h3, mask, y_part, hl_part, bal_counts, bal_lists;
  size_t dn_up, dn_gate, dn_a, dn_y2, dn_lt, total;  // dense fallback
};

constexpr size_t kLtWorkspace = 16u << 20;  // cuBLASLt workspace of the dense fallback

WsLayout layout(const sffn_layer* L, int batch) {
  const auto& d = L->desc;
  WsLayout w{};
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off = align_up(off + bytes, 256);
    return o;
  };
  w.hdr = take(sizeof(WsHeader));
  w.flags = take(barrier_flag_bytes((uint32_t)L->gather_grid));
  w.tickets = take((size_t)L->RG * batch * sizeof(uint32_t));
  w.h_part = take((size_t)std::max(std::max(L->KS, L->KS32), L->KStok) * batch * d.rank * sizeof(float));
  w.h = take((size_t)batch * d.rank * sizeof(float));
  w.h3 = take(L->esize == 2 ? (size_t)96 * d.rank * 2 : 0);  // h as three 16-bit parts, up to 32 tokens
  w.mask = take((size_t)batch * L->W * sizeof(uint32_t));
  w.y_part = take((size_t)L->gather_grid * std::min(batch, L->max_bt) * d.d_model * sizeof(float));
  w.hl_part = take(L->lcfg_ok ? layer_slot_bytes(d.rank) : 0);
  const size_t own_cap = (size_t)(d.d_ff + L->gather_grid - 1) / L->gather_grid;
  const int lg = std::max(L->gather_grid, L->layer_grid);
  const size_t lown_cap = L->layer_grid > 0 ? (size_t)(d.d_ff + L->layer_grid - 1) / L->layer_grid : own_cap;
  w.bal_counts = take(L->lcfg_ok ? (size_t)lg * sizeof(uint64_t) : 0);
  w.bal_lists = take(L->lcfg_ok ? (size_t)lg * std::max(own_cap, lown_cap) * 2 * sizeof(int32_t) : 0);
  const bool dn = L->dense_for(batch);
  w.dn_up = take(dn ? (size_t)batch * d.d_ff * sizeof(float) : 0);
  w.dn_gate = take(dn && d.act == SFFN_REGLU ? (size_t)batch * d.d_ff * sizeof(float) : 0);
  w.dn_a = take(dn ? (size_t)2 * batch * d.d_ff * L->esize : 0);
  w.dn_y2 = take(dn ? (size_t)2 * batch * d.d_model * sizeof(float) : 0);
  w.dn_lt = take(dn ? kLtWorkspace : 0);
  w.total = off;
  return w;
}

struct Ws {
  WsLayout lay;
  unsigned char* base;
  WsHeader* hdr() const { return reinterpret_cast<WsHeader*>(base + lay.hdr); }
  uint32_t* flags() const { return reinterpret_cast<uint32_t*>(base + lay.flags); }
  uint32_t* tickets() const { return reinterpret_cast<uint32_t*>(base + lay.tickets); }
  float* h_part() const { return reinterpret_cast<float*>(base + lay.h_part); }
  float* h() const { return reinterpret_cast<float*>(base + lay.h); }
  void* h3() const { return base + lay.h3; }
  uint32_t* mask() const { return reinterpret_cast<uint32_t*>(base + lay.mask); }
  float* y_part() const { return reinterpret_cast<float*>(base + lay.y_part); }
  unsigned long long* hl_slots() const { return reinterpret_cast<unsigned long long*>(base + lay.hl_part); }
  uint64_t* bal_counts() const { return reinterpret_cast<uint64_t*>(base + lay.bal_counts); }
  int32_t* bal_lists() const { return reinterpret_cast<int32_t*>(base + lay.bal_lists); }
  float* dn_up() const { return reinterpret_cast<float*>(base + lay.dn_up); }
  float* dn_gate() const { return reinterpret_cast<float*>(base + lay.dn_gate); }
  void* dn_a() const { return base + lay.dn_a; }
  float* dn_y2() const { return reinterpret_cast<float*>(base + lay.dn_y2); }
  void* dn_lt() const { return base + lay.dn_lt; }
};

sffn_status check_ws(const sffn_layer* L, int batch, void* ws, size_t bytes, Ws* out) {
  if (ws == nullptr) return fail(SFFN_ERR_WORKSPACE, "workspace is NULL");
  if ((reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return fail(SFFN_ERR_WORKSPACE, "workspace not 256-byte aligned");
  out->lay = layout(L, batch);
  if (bytes < out->lay.total)
    return fail(SFFN_ERR_WORKSPACE, "workspace too small: %zu bytes given, %zu needed", bytes, out->lay.total);
  out->base = static_cast<unsigned char*>(ws);
  return SFFN_OK;
}

sffn_status check_batch(const sffn_layer* L, int batch) {
  if (batch < 1 || batch > L->desc.max_batch)
    return fail(SFFN_ERR_INVALID_ARG, "batch %d outside [1, max_batch=%d]", batch, L->desc.max_batch);
  return SFFN_OK;
}

sffn_status check_dev_ptr(const void* p, const char* name) {
  if (p == nullptr) return fail(SFFN_ERR_INVALID_ARG, "%s is NULL", name);
  if (!aligned16(p)) return fail(SFFN_ERR_INVALID_ARG, "%s is not 16-byte aligned", name);
  return SFFN_OK;
}

#define SFFN_TRY(expr)                     \
  do {                                     \
    sffn_status _st = (expr);              \
    if (_st != SFFN_OK) return _st;        \
  } while (0)

#define SFFN_CUDA(expr, where)                          \
  do {                                                  \
    cudaError_t _e = (expr);                            \
    if (_e != cudaSuccess) return cuda_fail(_e, where); \
  } while (0)

// Predictor for `batch` tokens: h = V x (split-K, deterministic), then the
// scores and the mask words (and optionally the scores themselves).
bool use_union(const sffn_layer* L, int batch, UnionConfig* cfg);

sffn_status run_predictor(const sffn_layer* L, const void* x, int batch, const Ws& ws, float* scores,
                          cudaStream_t s) {
  const auto& d = L->desc;
  size_t ring = 0;
  UnionConfig uc{};
  if (scores == nullptr && use_union(L, batch, &uc) && score_mma_config(d.dtype, d.rank, batch, L->smem_optin, &ring)) {
    // one hidden-layer launch for the whole batch (h also as three 16-bit
    // parts), then the scores and threshold as one tensor-core product
    const int bt = batch <= 8 ? 8 : batch <= 16 ? 16 : 32;
    // the cluster kernel where d splits into its eighths; otherwise, above
    // 16 tokens the lane-per-token kernel (K-chunks of 256), below it the
    // token-group kernel
    const bool tok = batch > 16;
    PredHiddenArgs ha{d.pred_V, x, batch, d.rank, d.d_model, tok ? 256 : L->kc32, tok ? L->KStok : L->KS32,
                      ws.h_part(), ws.h(), ws.tickets(), ws.h3(), bt};
    const size_t hc = pred_hidden_cluster_smem(d.d_model, bt);
    ha.cluster = hc > 0 && hc <= L->smem_optin ? 1 : 0;
    SFFN_CUDA(launch_pred_hidden(d.dtype, ha, s), "predictor hidden launch");
    ScoreMmaArgs sa{d.pred_U, ws.h3(), d.pred_b, d.tau, batch, d.d_ff, d.rank, L->W, ws.mask(), ws.hdr(), ring,
                    (uint64_t)g_wait_ns};
    SFFN_CUDA(launch_score_mma(d.dtype, sa, bt, std::min(L->sms, L->W), s), "predictor score launch");
    return SFFN_OK;
  }
  PredHiddenArgs ha{d.pred_V, x, batch, d.rank, d.d_model, L->kc_elems, L->KS, ws.h_part(), ws.h(), ws.tickets(),
                    nullptr, 0};
  // token groups of up to 8 per launch
  for (int b0 = 0; b0 < batch; b0 += 8) {
    const int nb = std::min(8, batch - b0);
    PredHiddenArgs a = ha;
    a.x = static_cast<const unsigned char*>(x) + (size_t)b0 * d.d_model * L->esize;
    a.B = nb;
    a.h_part = ws.h_part() + (size_t)b0 * L->KS * d.rank;
    a.h = ws.h() + (size_t)b0 * d.rank;
    SFFN_CUDA(launch_pred_hidden(d.dtype, a, s), "predictor hidden launch");
    PredScoreArgs sa{d.pred_U, a.h, d.pred_b, d.tau, nb, d.d_ff, d.rank, L->W,
                     ws.mask() + (size_t)b0 * L->W,
                     scores ? scores + (size_t)b0 * d.d_ff : nullptr, L->score_grid};
    SFFN_CUDA(launch_pred_score(d.dtype, sa, s), "predictor score launch");
  }
  return SFFN_OK;
}

// Timing events must become graph nodes when the stream is being captured.
sffn_status record_profile_event(cudaEvent_t ev, cudaStream_t s) {
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  SFFN_CUDA(cudaStreamIsCapturing(s, &cs), "capture query");
  const unsigned flags = cs == cudaStreamCaptureStatusActive ? cudaEventRecordExternal : cudaEventRecordDefault;
  SFFN_CUDA(cudaEventRecordWithFlags(ev, s, flags), "profile event");
  return SFFN_OK;
}

// The profiling pair of the next dominant-kernel launch, if any is left.
bool profile_pair(cudaEvent_t* start, cudaEvent_t* stop) {
  if (g_prof_next >= g_prof_start.size()) return false;
  *start = g_prof_start[g_prof_next];
  *stop = g_prof_stop[g_prof_next];
  ++g_prof_next;
  return true;
}

// Gather passes of up to max_bt tokens each.
sffn_status run_gather(const sffn_layer* L, const void* x, int batch, float* y, const Ws& ws, bool dense,
                       cudaStream_t s) {
  const auto& d = L->desc;
  for (int b0 = 0; b0 < batch; b0 += L->max_bt) {
    const int nb = std::min(L->max_bt, batch - b0);
    const int bt = nb == 1 ? 1 : nb == 2 ? 2 : 4;
    if (!L->gcfg_ok[bt_slot(bt)]) return fail(SFFN_ERR_UNSUPPORTED, "no gather configuration for %d tokens", bt);
    GatherArgs a{};
    a.x = static_cast<const unsigned char*>(x) + (size_t)b0 * d.d_model * L->esize;
    a.w_up = d.w_up;
    a.w_gate = d.w_gate;
    a.w_downT = d.w_downT;
    a.b = d.b;
    a.mask = ws.mask() + (size_t)b0 * L->W;
    a.y = y + (size_t)b0 * d.d_model;
    a.y_part = ws.y_part();
    a.hdr = ws.hdr();
    a.bar_flags = ws.flags();
    a.B = nb;
    a.d = d.d_model;
    a.f = d.d_ff;
    a.W = L->W;
    a.act = d.act;
    a.dense = dense ? 1 : 0;
    a.nstages = L->gcfg[bt_slot(bt)].nstages;
    a.list_cap = L->gcfg[bt_slot(bt)].list_cap;
    a.wait_ns = (uint64_t)g_wait_ns;
    a.wstride = L->wstride;
    cudaEvent_t e0, e1;
    const bool prof = profile_pair(&e0, &e1);
    if (prof) SFFN_TRY(record_profile_event(e0, s));
    SFFN_CUDA(launch_gather(d.dtype, L->gcfg[bt_slot(bt)], a, L->gather_grid, s), "gather launch");
    if (prof) SFFN_TRY(record_profile_event(e1, s));
  }
  return SFFN_OK;
}

// Batches this large (and 16-bit weights) go to the tensor-core union path
// (measured on the ReGLU layer: at 2 tokens the row gather is faster, at 4
// the union path is 1.2x faster, at 6 2x).
constexpr int kUnionMinBatch = 3;

bool use_union(const sffn_layer* L, int batch, UnionConfig* cfg) {
  const auto& d = L->desc;
  if (batch < kUnionMinBatch || (d.flags & SFFN_FLAG_ROW_GATHER)) return false;
  return union_config(d.dtype, d.act, d.d_model, d.d_ff, batch, L->gather_grid, L->smem_optin, cfg);
}

// The dense fallback's cuBLASLt plan for `batch` tokens, built on first use
// (host-side descriptors and a heuristic query only).
sffn_status dense_plan(sffn_layer* L, int batch, DensePlan** out) {
  DensePlan& p = L->plans[batch];
  *out = &p;
  if (p.built) return p.ok ? SFFN_OK : fail(SFFN_ERR_UNSUPPORTED, "no cuBLASLt algorithm for the dense fallback");
  p.built = true;
  const auto& d = L->desc;
  const cudaDataType_t wt = d.dtype == SFFN_BF16 ? CUDA_R_16BF : CUDA_R_16F;
  const uint64_t ldw = L->wstride / L->esize;
  const cublasOperation_t opT = CUBLAS_OP_T, opN = CUBLAS_OP_N;
  bool ok = cublasLtMatmulDescCreate(&p.op1, CUBLAS_COMPUTE_32F, CUDA_R_32F) == CUBLAS_STATUS_SUCCESS &&
            cublasLtMatmulDescSetAttribute(p.op1, CUBLASLT_MATMUL_DESC_TRANSA, &opT, sizeof(opT)) ==
                CUBLAS_STATUS_SUCCESS &&
            cublasLtMatmulDescSetAttribute(p.op1, CUBLASLT_MATMUL_DESC_TRANSB, &opN, sizeof(opN)) ==
                CUBLAS_STATUS_SUCCESS &&
            cublasLtMatmulDescCreate(&p.op2, CUBLAS_COMPUTE_32F, CUDA_R_32F) == CUBLAS_STATUS_SUCCESS &&
            // column-major views of the row-major arrays:
            // W (d x f, ld ldw), X (d x B), D (f x B); W_down^T (d x f), A (f x 2B), Y2 (d x 2B)
            cublasLtMatrixLayoutCreate(&p.w1, wt, d.d_model, d.d_ff, ldw) == CUBLAS_STATUS_SUCCESS &&
            cublasLtMatrixLayoutCreate(&p.x1, wt, d.d_model, batch, d.d_model) == CUBLAS_STATUS_SUCCESS &&
            cublasLtMatrixLayoutCreate(&p.d1, CUDA_R_32F, d.d_ff, batch, d.d_ff) == CUBLAS_STATUS_SUCCESS &&
            cublasLtMatrixLayoutCreate(&p.w2, wt, d.d_model, d.d_ff, ldw) == CUBLAS_STATUS_SUCCESS &&
            cublasLtMatrixLayoutCreate(&p.a2, wt, d.d_ff, 2 * batch, d.d_ff) == CUBLAS_STATUS_SUCCESS &&
            cublasLtMatrixLayoutCreate(&p.y2, CUDA_R_32F, d.d_model, 2 * batch, d.d_model) == CUBLAS_STATUS_SUCCESS;
  cublasLtMatmulPreference_t pref = nullptr;
  if (ok) {
    const uint64_t wsb = kLtWorkspace;
    const uint32_t align = 16;  // tokens may start on any 16-byte boundary
    ok = cublasLtMatmulPreferenceCreate(&pref) == CUBLAS_STATUS_SUCCESS &&
         cublasLtMatmulPreferenceSetAttribute(pref, CUBLASLT_MATMUL_PREF_MAX_WORKSPACE_BYTES, &wsb, sizeof(wsb)) ==
             CUBLAS_STATUS_SUCCESS;
    for (auto attr : {CUBLASLT_MATMUL_PREF_MIN_ALIGNMENT_A_BYTES, CUBLASLT_MATMUL_PREF_MIN_ALIGNMENT_B_BYTES,
                      CUBLASLT_MATMUL_PREF_MIN_ALIGNMENT_C_BYTES, CUBLASLT_MATMUL_PREF_MIN_ALIGNMENT_D_BYTES})
      ok = ok && cublasLtMatmulPreferenceSetAttribute(pref, attr, &align, sizeof(align)) == CUBLAS_STATUS_SUCCESS;
  }
  if (ok) {
    cublasLtMatmulHeuristicResult_t r1{}, r2{};
    int n1 = 0, n2 = 0;
    ok = cublasLtMatmulAlgoGetHeuristic(L->lt, p.op1, p.w1, p.x1, p.d1, p.d1, pref, 1, &r1, &n1) ==
             CUBLAS_STATUS_SUCCESS && n1 > 0 &&
         cublasLtMatmulAlgoGetHeuristic(L->lt, p.op2, p.w2, p.a2, p.y2, p.y2, pref, 1, &r2, &n2) ==
             CUBLAS_STATUS_SUCCESS && n2 > 0;
    if (ok) {
      p.algo1 = r1.algo;
      p.algo2 = r2.algo;
    }
  }
  if (pref) cublasLtMatmulPreferenceDestroy(pref);
  p.ok = ok;
  return ok ? SFFN_OK : fail(SFFN_ERR_UNSUPPORTED, "no cuBLASLt algorithm for the dense fallback");
}

// Dense fallback: every row of the layer through two tensor-core GEMMs, the
// tokens' masks applied between them (dense.cu).
sffn_status run_dense_ffn(const sffn_layer* Lc, const void* x, int batch, float* y, const Ws& ws, cudaStream_t s) {
  sffn_layer* L = const_cast<sffn_layer*>(Lc);  // plans are built lazily
  const auto& d = L->desc;
  DensePlan* p = nullptr;
  SFFN_TRY(dense_plan(L, batch, &p));
  const float one = 1.f, zero = 0.f;
  auto gemm1 = [&](const void* w, float* out) {
    return cublasLtMatmul(L->lt, p->op1, &one, w, p->w1, x, p->x1, &zero, out, p->d1, out, p->d1, &p->algo1,
                          ws.dn_lt(), kLtWorkspace, s);
  };
  if (gemm1(d.w_up, ws.dn_up()) != CUBLAS_STATUS_SUCCESS)
    return fail(SFFN_ERR_CUDA, "dense fallback: up GEMM failed");
  if (d.act == SFFN_REGLU && gemm1(d.w_gate, ws.dn_gate()) != CUBLAS_STATUS_SUCCESS)
    return fail(SFFN_ERR_CUDA, "dense fallback: gate GEMM failed");
  SFFN_CUDA(launch_dense_act(d.dtype, ws.dn_up(), d.act == SFFN_REGLU ? ws.dn_gate() : nullptr, d.b, ws.mask(), batch,
                             d.d_ff, L->W, ws.dn_a(), s),
            "dense activation launch");
  if (cublasLtMatmul(L->lt, p->op2, &one, d.w_downT, p->w2, ws.dn_a(), p->a2, &zero, ws.dn_y2(), p->y2, ws.dn_y2(),
                     p->y2, &p->algo2, ws.dn_lt(), kLtWorkspace, s) != CUBLAS_STATUS_SUCCESS)
    return fail(SFFN_ERR_CUDA, "dense fallback: down GEMM failed");
  SFFN_CUDA(launch_dense_combine(ws.dn_y2(), batch, d.d_model, y, s), "dense combine launch");
  return SFFN_OK;
}

// The sparse products of a batch whose mask words are in the workspace.
sffn_status run_sparse_ffn(const sffn_layer* L, const void* x, int batch, float* y, const Ws& ws, cudaStream_t s) {
  if (L->dense_for(batch)) return run_dense_ffn(L, x, batch, y, ws, s);
  UnionConfig uc{};
  if (!use_union(L, batch, &uc)) return run_gather(L, x, batch, y, ws, false, s);
  const auto& d = L->desc;
  SFFN_CUDA(cudaMemsetAsync(y, 0, (size_t)batch * d.d_model * sizeof(float), s), "output clear");
  UnionArgs a{};
  a.x = x;
  a.w_up = d.w_up;
  a.w_gate = d.w_gate;
  a.w_downT = d.w_downT;
  a.b = d.b;
  a.mask = ws.mask();
  a.y = y;
  a.hdr = ws.hdr();
  a.B = batch;
  a.d = d.d_model;
  a.f = d.d_ff;
  a.W = L->W;
  a.act = d.act;
  a.list_cap = uc.list_cap;
  a.ring_bytes = uc.ring_bytes;
  a.wait_ns = (uint64_t)g_wait_ns;
  a.wstride = L->wstride;
  cudaEvent_t e0, e1;
  const bool prof = profile_pair(&e0, &e1);
  if (prof) SFFN_TRY(record_profile_event(e0, s));
  SFFN_CUDA(launch_union(d.dtype, uc, a, L->gather_grid, s), "union launch");
  if (prof) SFFN_TRY(record_profile_event(e1, s));
  return SFFN_OK;
}

sffn_status check_x(const sffn_layer* L, const void* x) { return check_dev_ptr(x, "x"); }

// One token through the single-launch layer kernel.  With y_prev, the kernel
// first forms x = round(LN(x_prev + y_prev)) and stores it at x_ln_out.
// Look-ahead stacks: the call's own rows come from la_in and the predictor of
// `pred` (the next layer) is evaluated into la_out; predict_only runs only
// that predictor (no rows, no y, launched without clusters).
struct LookAhead {
  const sffn_layer* pred = nullptr;
  const uint32_t* la_in = nullptr;
  uint32_t* la_out = nullptr;
  bool predict_only = false;
};

sffn_status run_layer(const sffn_layer* L, const void* x, const float* y_prev, void* x_ln_out, const float* gamma,
                      const float* beta, float eps, float* y, uint32_t* mask, const Ws& ws, cudaStream_t s,
                      const LookAhead& la = LookAhead()) {
  const auto& d = L->desc;
  const auto& pd = la.pred != nullptr ? la.pred->desc : L->desc;  // the predictor this launch evaluates
  LayerArgs a{};
  a.x = x;
  a.y_prev = y_prev;
  a.x_ln_out = x_ln_out;
  a.ln_gamma = gamma;
  a.ln_beta = beta;
  a.ln_eps = eps;
  a.V = pd.pred_V;
  a.U = pd.pred_U;
  a.pb = pd.pred_b;
  a.b = d.b;
  a.tau = pd.tau;
  a.w_up = d.w_up;
  a.w_gate = d.w_gate;
  a.w_downT = d.w_downT;
  a.y = y;
  a.h_slots = ws.hl_slots();
  a.mask = mask;
  a.la_in = la.la_in;
  a.la_out = la.la_out;
  a.predict_only = la.predict_only ? 1 : 0;
  a.hdr = ws.hdr();
  a.bar_flags = ws.flags();
  a.d = d.d_model;
  a.f = d.d_ff;
  a.r = d.rank;
  a.act = d.act;
  a.nstages = L->lcfg.nstages;
  a.u_smem = L->lcfg.u_smem;
  a.region_bytes = L->lcfg.region_bytes;
  a.u_off = L->lcfg.u_off;
  a.hot_rows = d.hot_rows;
  a.warm_rows = d.warm_rows;
  a.hot_stages = L->lcfg.hot_stages;
  const int own_cap = (d.d_ff + L->layer_grid - 1) / L->layer_grid;
  // the balancing exchange holds at most 256 block counts
  a.balance = L->lcfg.balance && own_cap >= 8 && L->layer_grid <= 256 && la.pred == nullptr ? 1 : 0;
  a.cluster = a.balance == 0 && !la.predict_only ? L->layer_cluster : 0;
  a.static_weights = (d.flags & SFFN_FLAG_STATIC_WEIGHTS) ? 1 : 0;
  int prefill = L->lcfg.hot_stages;
  if (d.expected_active > 0.f)
    prefill = std::max(prefill, std::min(L->lcfg.nstages, (int)(0.85f * d.expected_active / L->layer_grid)));
  a.prefill = prefill;
  a.bal_counts = ws.bal_counts();
  a.bal_lists = ws.bal_lists();
  a.wait_ns = (uint64_t)g_wait_ns;
  a.wstride = L->wstride;
  cudaEvent_t e0, e1;
  const bool prof = profile_pair(&e0, &e1);
  if (prof) SFFN_TRY(record_profile_event(e0, s));
  SFFN_CUDA(launch_layer(d.dtype, L->lcfg, a, L->layer_grid, s), "layer launch");
  if (prof) SFFN_TRY(record_profile_event(e1, s));
  return SFFN_OK;
}

}  // namespace

extern "C" {

int32_t sffn_version(void) { return kVersion; }

const char* sffn_last_error(void) { return g_err.c_str(); }

const char* sffn_status_string(sffn_status st) {
  switch (st) {
    case SFFN_OK: return "ok";
    case SFFN_ERR_INVALID_ARG: return "invalid argument";
    case SFFN_ERR_UNSUPPORTED: return "unsupported";
    case SFFN_ERR_CUDA: return "CUDA error";
    case SFFN_ERR_CAPACITY: return "capacity exceeded";
    case SFFN_ERR_TIMEOUT: return "device wait timed out";
    case SFFN_ERR_WORKSPACE: return "bad workspace";
  }
  return "unknown status";
}

sffn_status sffn_set_profile_events(void* const* start_events, void* const* stop_events, int32_t n_pairs) {
  g_err.clear();
  if (n_pairs < 0 || (n_pairs > 0 && (start_events == nullptr || stop_events == nullptr)))
    return fail(SFFN_ERR_INVALID_ARG, "profile events: %d pairs, arrays NULL", n_pairs);
  g_prof_start.clear();
  g_prof_stop.clear();
  for (int i = 0; i < n_pairs; ++i) {
    if (start_events[i] == nullptr || stop_events[i] == nullptr)
      return fail(SFFN_ERR_INVALID_ARG, "profile event pair %d is NULL", i);
    g_prof_start.push_back(static_cast<cudaEvent_t>(start_events[i]));
    g_prof_stop.push_back(static_cast<cudaEvent_t>(stop_events[i]));
  }
  g_prof_next = 0;
  return SFFN_OK;
}

sffn_status sffn_set_wait_limit_ns(int64_t ns) {
  if (ns <= 0) return fail(SFFN_ERR_INVALID_ARG, "wait limit must be positive");
  g_wait_ns = ns;
  return SFFN_OK;
}

sffn_status sffn_create_layer(const sffn_layer_desc* desc, sffn_layer_t* out) {
  g_err.clear();
  if (desc == nullptr || out == nullptr) return fail(SFFN_ERR_INVALID_ARG, "desc/out is NULL");
  *out = nullptr;
  const sffn_layer_desc& d = *desc;
  if (d.dtype != SFFN_F32 && d.dtype != SFFN_F16 && d.dtype != SFFN_BF16)
    return fail(SFFN_ERR_INVALID_ARG, "unknown dtype %d", d.dtype);
  if (d.act != SFFN_RELU && d.act != SFFN_REGLU) return fail(SFFN_ERR_INVALID_ARG, "unknown act %d", d.act);
  if (d.d_model <= 0 || d.d_ff <= 0 || d.rank <= 0)
    return fail(SFFN_ERR_INVALID_ARG, "d_model, d_ff and rank must be positive");
  if (d.max_batch < 1 || d.max_batch > 32) return fail(SFFN_ERR_INVALID_ARG, "max_batch must be in [1, 32]");
  if (d.flags & ~(SFFN_FLAG_MULTI_KERNEL | SFFN_FLAG_BALANCE | SFFN_FLAG_ROW_GATHER | SFFN_FLAG_STATIC_WEIGHTS |
                  SFFN_FLAG_BUNDLED))
    return fail(SFFN_ERR_INVALID_ARG, "unknown flag bits 0x%x", (unsigned)d.flags);
  const int esize = d.dtype == SFFN_F32 ? 4 : 2;
  if (((size_t)d.d_model * esize) % 16 != 0)
    return fail(SFFN_ERR_INVALID_ARG, "d_model * sizeof(dtype) must be a multiple of 16");
  if (((size_t)d.rank * esize) % 16 != 0)
    return fail(SFFN_ERR_INVALID_ARG, "rank * sizeof(dtype) must be a multiple of 16");
  SFFN_TRY(check_dev_ptr(d.w_up, "w_up"));
  SFFN_TRY(check_dev_ptr(d.pred_U, "pred_U"));
  SFFN_TRY(check_dev_ptr(d.pred_V, "pred_V"));
  if (d.pred_b == nullptr) return fail(SFFN_ERR_INVALID_ARG, "pred_b is NULL");
  const bool bundled = (d.flags & SFFN_FLAG_BUNDLED) != 0;
  if (bundled) {
    if (d.w_gate != nullptr || d.w_downT != nullptr)
      return fail(SFFN_ERR_INVALID_ARG, "bundled layers pass the bundle as w_up; w_gate and w_downT must be NULL");
  } else {
    SFFN_TRY(check_dev_ptr(d.w_downT, "w_downT"));
    if (d.act == SFFN_REGLU) {
      SFFN_TRY(check_dev_ptr(d.w_gate, "w_gate"));
    } else if (d.w_gate != nullptr) {
      return fail(SFFN_ERR_INVALID_ARG, "w_gate must be NULL for ReLU layers");
    }
  }
  if (d.rank / (16 / esize) > 256) return fail(SFFN_ERR_UNSUPPORTED, "rank too large for the score kernel");
  if (d.hot_rows < 0 || d.hot_rows > d.d_ff) return fail(SFFN_ERR_INVALID_ARG, "hot_rows outside [0, d_ff]");
  if (d.warm_rows < 0 || d.warm_rows > d.d_ff) return fail(SFFN_ERR_INVALID_ARG, "warm_rows outside [0, d_ff]");
  if (!(d.expected_active >= 0.f)) return fail(SFFN_ERR_INVALID_ARG, "expected_active must be >= 0");
  if (d.dense_min_batch < 0 || d.dense_min_batch > 32)
    return fail(SFFN_ERR_INVALID_ARG, "dense_min_batch outside [0, 32]");
  if (d.dense_min_batch > 0 && (d.dtype == SFFN_F32 || d.dense_min_batch < 2))
    return fail(SFFN_ERR_UNSUPPORTED, "the dense fallback takes 16-bit weights and batches of 2 or more");

  sffn_layer* L = new (std::nothrow) sffn_layer();
  if (L == nullptr) return fail(SFFN_ERR_INVALID_ARG, "out of host memory");
  L->desc = d;
  L->esize = esize;
  L->wstride = (size_t)d.d_model * esize;
  if (bundled) {  // neuron i's rows side by side: [gate | up | down] (ReGLU) or [up | down] (ReLU)
    const unsigned char* bnd = static_cast<const unsigned char*>(d.w_up);
    const size_t rb = (size_t)d.d_model * esize;
    const int nm = d.act == SFFN_REGLU ? 2 : 1;
    L->wstride = (size_t)(nm + 1) * rb;
    L->desc.w_gate = d.act == SFFN_REGLU ? bnd : nullptr;
    L->desc.w_up = bnd + (size_t)(nm - 1) * rb;
    L->desc.w_downT = bnd + (size_t)nm * rb;
  }
  cudaError_t e = cudaGetDevice(&L->device);
  int optin = 0;
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&L->sms, cudaDevAttrMultiProcessorCount, L->device);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, L->device);
  if (e != cudaSuccess) {
    delete L;
    return cuda_fail(e, "device query");
  }
  L->smem_optin = (size_t)optin;
  L->W = (d.d_ff + 31) / 32;

  // predictor split: about two blocks per SM across (K-chunks x row groups)
  const int E = 16 / esize;
  const int unit = 32 * E;  // one warp-wide 16-byte load of a row
  L->RG = pred_hidden_row_groups(d.rank);
  const int rg16 = (d.rank + 15) / 16;  // row groups of the up-to-8-token kernel
  const int ks_target = std::max(1, (2 * L->sms + rg16 - 1) / rg16);
  int kc = (d.d_model + ks_target - 1) / ks_target;
  kc = (kc + unit - 1) / unit * unit;
  const int max_kc = 8192 / esize;  // x chunk of 8 tokens must stay within 64 KB of shared memory
  kc = std::min(kc, std::max(unit, max_kc / unit * unit));
  L->kc_elems = kc;
  L->KS = (d.d_model + kc - 1) / kc;
  const int max_kc32 = 2048 / esize;  // x chunk of 32 tokens must stay within 64 KB of shared memory
  L->kc32 = std::min(kc, std::max(unit, max_kc32 / unit * unit));
  L->KS32 = (d.d_model + L->kc32 - 1) / L->kc32;
  L->KStok = (d.d_model + 255) / 256;  // the lane-per-token kernel's K-chunks of 256
  L->score_grid = std::min((d.d_ff + 63) / 64, 8 * L->sms);

  L->gather_grid = L->sms;
  L->max_bt = gather_max_bt(d.dtype, d.d_model);
  if (L->max_bt == 0) {
    delete L;
    return fail(SFFN_ERR_UNSUPPORTED, "d_model %d too wide for the gather kernel", d.d_model);
  }
  for (int bt : {1, 2, 4}) {
    if (bt > L->max_bt) continue;
    L->gcfg_ok[bt_slot(bt)] =
        gather_config(d.dtype, d.act, d.d_model, d.d_ff, bt, L->gather_grid, L->smem_optin, &L->gcfg[bt_slot(bt)]);
  }
  if (!L->gcfg_ok[0]) {
    delete L;
    return fail(SFFN_ERR_UNSUPPORTED, "rows of d_model %d do not fit two pipeline stages", d.d_model);
  }
  while (!L->gcfg_ok[bt_slot(L->max_bt)]) L->max_bt /= 2;
  // The batch-1 layer kernel runs two blocks per SM when two fit with at
  // least kMinStages2 ring stages each (two copy rings per SM move more than
  // one: OPT-6.7B layer, six 16 KB stages, 17.9 us per layer against 19.3;
  // Llama-7B ReGLU layer, four 24 KB stages, 19.0 us against 19.9), else one;
  // every block waits for h values that other blocks
  // publish, so every block must be resident, which the occupancy query
  // confirms.  The balancing scratch takes shared memory only when asked for.
  {
    const bool balance = (d.flags & SFFN_FLAG_BALANCE) != 0;
    int smem_sm = 0;
    cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, L->device);
    const size_t half = smem_sm > 0 ? (size_t)smem_sm / 2 - 1024 - 3072 : 0;  // per-block reserve, static smem
    LayerConfig c2{};
    if (half > 0 && layer_config(d.dtype, d.act, d.d_model, d.d_ff, d.rank, 2 * L->sms, half, balance, &c2) &&
        c2.nstages >= kMinStages2 && layer_blocks_per_sm(d.dtype, c2) >= 2) {
      L->lcfg = c2;
      L->layer_grid = 2 * L->sms;
      L->lcfg_ok = true;
    } else {
      L->layer_grid = L->gather_grid;
      L->lcfg_ok = layer_config(d.dtype, d.act, d.d_model, d.d_ff, d.rank, L->layer_grid, L->smem_optin, balance,
                                &L->lcfg) &&
                   layer_blocks_per_sm(d.dtype, L->lcfg) >= 1;
    }
    // With one block per SM, pairs of blocks (clusters of two) split their
    // active rows evenly, when every pair fits at once (ReGLU layer 42.0K ->
    // 45.9K tokens/s; at two blocks per SM the exchange cost more than the
    // smaller spread of rows saved)
    L->layer_cluster = L->lcfg_ok && L->layer_grid == L->sms && L->layer_grid % 2 == 0 &&
                               layer_max_clusters(d.dtype, L->lcfg, L->layer_grid, 2) * 2 >= L->layer_grid
                           ? 2
                           : 0;
  }
  if (d.dense_min_batch > 0 && cublasLtCreate(&L->lt) != CUBLAS_STATUS_SUCCESS) {
    delete L;
    return fail(SFFN_ERR_CUDA, "cublasLtCreate failed");
  }
  *out = L;
  return SFFN_OK;
}

sffn_status sffn_destroy_layer(sffn_layer_t layer) {
  delete layer;
  return SFFN_OK;
}

sffn_status sffn_get_layer_info(sffn_layer_t L, sffn_layer_info* info) {
  g_err.clear();
  if (L == nullptr || info == nullptr) return fail(SFFN_ERR_INVALID_ARG, "layer or info is NULL");
  sffn_layer_info o{};
  o.fused = L->fused() ? 1 : 0;
  if (L->lcfg_ok) {
    o.grid = L->layer_grid;
    o.blocks_per_sm = L->sms > 0 ? L->layer_grid / L->sms : 0;
    o.cluster = L->layer_cluster;
    o.ring_stages = L->lcfg.nstages;
    o.hot_stages = L->lcfg.hot_stages;
  }
  if (!o.fused) o.grid = 0;
  *info = o;
  return SFFN_OK;
}

size_t sffn_workspace_size(sffn_layer_t L, int32_t batch) {
  if (L == nullptr || batch < 1 || batch > L->desc.max_batch) return 0;
  return layout(L, batch).total;
}

sffn_status sffn_workspace_init(void* ws, size_t bytes, void* stream) {
  if (ws == nullptr) return fail(SFFN_ERR_WORKSPACE, "workspace is NULL");
  SFFN_CUDA(cudaMemsetAsync(ws, 0, bytes, static_cast<cudaStream_t>(stream)), "workspace memset");
  return SFFN_OK;
}

sffn_status sffn_predict(sffn_layer_t L, const void* x, int32_t batch, int32_t* idx, int32_t* n_active,
                         void* workspace, size_t ws_bytes, void* stream) {
  g_err.clear();
  if (L == nullptr) return fail(SFFN_ERR_INVALID_ARG, "layer is NULL");
  SFFN_TRY(check_batch(L, batch));
  SFFN_TRY(check_x(L, x));
  if (idx == nullptr || n_active == nullptr) return fail(SFFN_ERR_INVALID_ARG, "idx/n_active is NULL");
  Ws ws;
  SFFN_TRY(check_ws(L, batch, workspace, ws_bytes, &ws));
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  SFFN_TRY(run_predictor(L, x, batch, ws, nullptr, s));
  SFFN_CUDA(launch_compact(ws.mask(), batch, L->desc.d_ff, L->W, idx, n_active, s), "compaction launch");
  return SFFN_OK;
}

sffn_status sffn_predict_scores(sffn_layer_t L, const void* x, int32_t batch, float* scores, void* workspace,
                                size_t ws_bytes, void* stream) {
  g_err.clear();
  if (L == nullptr) return fail(SFFN_ERR_INVALID_ARG, "layer is NULL");
  SFFN_TRY(check_batch(L, batch));
  SFFN_TRY(check_x(L, x));
  if (scores == nullptr) return fail(SFFN_ERR_INVALID_ARG, "scores is NULL");
  Ws ws;
  SFFN_TRY(check_ws(L, batch, workspace, ws_bytes, &ws));
  return run_predictor(L, x, batch, ws, scores, static_cast<cudaStream_t>(stream));
}

sffn_status sffn_forward(sffn_layer_t L, const void* x, int32_t batch, float* y, int32_t* idx_out,
                         int32_t* n_active_out, void* workspace, size_t ws_bytes, void* stream) {
  g_err.clear();
  if (L == nullptr) return fail(SFFN_ERR_INVALID_ARG, "layer is NULL");
  SFFN_TRY(check_batch(L, batch));
  SFFN_TRY(check_x(L, x));
  SFFN_TRY(check_dev_ptr(y, "y"));
  if ((idx_out == nullptr) != (n_active_out == nullptr))
    return fail(SFFN_ERR_INVALID_ARG, "idx_out and n_active_out must both be given or both be NULL");
  Ws ws;
  SFFN_TRY(check_ws(L, batch, workspace, ws_bytes, &ws));
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (batch == 1 && L->fused()) {
    SFFN_TRY(run_layer(L, x, nullptr, nullptr, nullptr, nullptr, 0.f, y, idx_out ? ws.mask() : nullptr, ws, s));
    if (idx_out != nullptr)
      SFFN_CUDA(launch_compact(ws.mask(), 1, L->desc.d_ff, L->W, idx_out, n_active_out, s), "compaction launch");
    return SFFN_OK;
  }
  SFFN_TRY(run_predictor(L, x, batch, ws, nullptr, s));
  if (idx_out != nullptr)
    SFFN_CUDA(launch_compact(ws.mask(), batch, L->desc.d_ff, L->W, idx_out, n_active_out, s), "compaction launch");
  return run_sparse_ffn(L, x, batch, y, ws, s);
}

sffn_status sffn_dense_forward(sffn_layer_t L, const void* x, int32_t batch, float* y, void* workspace,
                               size_t ws_bytes, void* stream) {
  g_err.clear();
  if (L == nullptr) return fail(SFFN_ERR_INVALID_ARG, "layer is NULL");
  SFFN_TRY(check_batch(L, batch));
  SFFN_TRY(check_x(L, x));
  SFFN_TRY(check_dev_ptr(y, "y"));
  Ws ws;
  SFFN_TRY(check_ws(L, batch, workspace, ws_bytes, &ws));
  return run_gather(L, x, batch, y, ws, true, static_cast<cudaStream_t>(stream));
}

sffn_status sffn_residual_layernorm(const void* x, const float* y, int32_t batch, int32_t d_model, int32_t dtype,
                                    const float* gamma, const float* beta, float eps, void* x_out, void* stream) {
  g_err.clear();
  if (dtype != SFFN_F32 && dtype != SFFN_F16 && dtype != SFFN_BF16)
    return fail(SFFN_ERR_INVALID_ARG, "unknown dtype %d", dtype);
  const int esize = dtype == SFFN_F32 ? 4 : 2;
  if (batch < 1 || d_model <= 0 || ((size_t)d_model * esize) % 16 != 0)
    return fail(SFFN_ERR_INVALID_ARG, "bad batch/d_model");
  if (!(eps >= 0.f)) return fail(SFFN_ERR_INVALID_ARG, "eps must be >= 0");
  SFFN_TRY(check_dev_ptr(x, "x"));
  SFFN_TRY(check_dev_ptr(y, "y"));
  SFFN_TRY(check_dev_ptr(x_out, "x_out"));
  SFFN_CUDA(launch_residual_layernorm(dtype, x, y, batch, d_model, gamma, beta, eps, x_out,
                                      static_cast<cudaStream_t>(stream)),
            "layernorm launch");
  return SFFN_OK;
}

size_t sffn_stack_workspace_size(const sffn_layer_t* layers, int32_t n_layers, int32_t batch) {
  if (layers == nullptr || n_layers < 1) return 0;
  size_t per = 0;
  for (int l = 0; l < n_layers; ++l) {
    const size_t w = sffn_workspace_size(layers[l], batch);
    if (w == 0) return 0;
    per = std::max(per, w);
  }
  const auto& d = layers[0]->desc;
  const size_t xb = align_up((size_t)batch * d.d_model * layers[0]->esize, 256);
  const size_t yb = align_up((size_t)batch * d.d_model * sizeof(float), 256);
  int Wmax = 0;
  for (int l = 0; l < n_layers; ++l) Wmax = std::max(Wmax, layers[l]->W);
  const size_t lab = align_up((size_t)Wmax * sizeof(uint32_t), 256);  // look-ahead mask words, two buffers
  return align_up(per, 256) + 2 * xb + 2 * yb + 2 * lab;
}

// Whether a stack can run with look-ahead masks: batch 1, every layer on the
// single-launch kernel with the same shapes and launch configuration (block
// c owns the same neurons in every layer, and the U-row staging of the next
// layer's predictor fits this layer's shared-memory plan), no balancing.
static sffn_status check_lookahead(const sffn_layer_t* layers, int n_layers, int batch) {
  if (batch != 1) return fail(SFFN_ERR_UNSUPPORTED, "look-ahead masks are built for batch 1 only");
  const sffn_layer* L0 = layers[0];
  for (int l = 0; l < n_layers; ++l) {
    const sffn_layer* L = layers[l];
    if (!L->fused() || (L->desc.flags & SFFN_FLAG_BALANCE))
      return fail(SFFN_ERR_UNSUPPORTED, "look-ahead: layer %d does not run the single-launch kernel without balancing", l);
    const auto &a = L->desc, &b = L0->desc;
    if (a.d_ff != b.d_ff || a.rank != b.rank || a.act != b.act || L->layer_grid != L0->layer_grid ||
        L->layer_cluster != L0->layer_cluster || L->lcfg.nstages != L0->lcfg.nstages ||
        L->lcfg.u_smem != L0->lcfg.u_smem || L->lcfg.u_off != L0->lcfg.u_off ||
        L->lcfg.region_bytes != L0->lcfg.region_bytes || L->lcfg.hot_stages != L0->lcfg.hot_stages)
      return fail(SFFN_ERR_UNSUPPORTED, "look-ahead: layer %d differs in shape or launch configuration", l);
  }
  return SFFN_OK;
}

sffn_status sffn_forward_stack(const sffn_layer_t* layers, int32_t n_layers, const void* x0, int32_t batch,
                               int32_t n_steps, void* x_out, void* x_trace, uint32_t* mask_trace,
                               float* y_trace, const float* ln_gamma, const float* ln_beta, float ln_eps,
                               int32_t options, void* workspace, size_t ws_bytes, void* stream) {
  g_err.clear();
  if (layers == nullptr || n_layers < 1) return fail(SFFN_ERR_INVALID_ARG, "no layers");
  if (n_steps < 1) return fail(SFFN_ERR_INVALID_ARG, "n_steps must be >= 1");
  for (int l = 0; l < n_layers; ++l) {
    if (layers[l] == nullptr) return fail(SFFN_ERR_INVALID_ARG, "layer %d is NULL", l);
    SFFN_TRY(check_batch(layers[l], batch));
    if (layers[l]->desc.d_model != layers[0]->desc.d_model || layers[l]->desc.dtype != layers[0]->desc.dtype)
      return fail(SFFN_ERR_INVALID_ARG, "layer %d differs in d_model or dtype", l);
  }
  SFFN_TRY(check_dev_ptr(x0, "x0"));
  SFFN_TRY(check_dev_ptr(x_out, "x_out"));
  if (x_trace != nullptr) SFFN_TRY(check_dev_ptr(x_trace, "x_trace"));
  if (mask_trace != nullptr) SFFN_TRY(check_dev_ptr(mask_trace, "mask_trace"));
  if (y_trace != nullptr) SFFN_TRY(check_dev_ptr(y_trace, "y_trace"));
  if (!(ln_eps >= 0.f)) return fail(SFFN_ERR_INVALID_ARG, "ln_eps must be >= 0");
  if (options & ~SFFN_STACK_LOOKAHEAD) return fail(SFFN_ERR_INVALID_ARG, "unknown option bits 0x%x", (unsigned)options);
  const bool lookahead = (options & SFFN_STACK_LOOKAHEAD) != 0;
  if (lookahead) SFFN_TRY(check_lookahead(layers, n_layers, batch));
  const size_t need = sffn_stack_workspace_size(layers, n_layers, batch);
  if (workspace == nullptr || ws_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return fail(SFFN_ERR_WORKSPACE, "stack workspace: %zu bytes needed (256-byte aligned)", need);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const auto& d0 = layers[0]->desc;
  const int esize = layers[0]->esize;
  size_t per = 0;
  for (int l = 0; l < n_layers; ++l) per = std::max(per, sffn_workspace_size(layers[l], batch));
  per = align_up(per, 256);
  unsigned char* base = static_cast<unsigned char*>(workspace);
  const size_t xbytes = (size_t)batch * d0.d_model * esize;
  const size_t xb = align_up(xbytes, 256);
  unsigned char* xbuf[2] = {base + per, base + per + xb};
  const size_t yb = align_up((size_t)batch * d0.d_model * sizeof(float), 256);
  float* ybufs[2] = {reinterpret_cast<float*>(base + per + 2 * xb), reinterpret_cast<float*>(base + per + 2 * xb + yb)};
  float* ybuf = ybufs[0];
  unsigned char* trace = static_cast<unsigned char*>(x_trace);
  unsigned char* xo = static_cast<unsigned char*>(x_out);
  // traces of every layer call: mask words (Wmax per token, the widest
  // layer's count) and outputs; a traced call writes its output in place
  int Wmax = 0;
  for (int l = 0; l < n_layers; ++l) Wmax = std::max(Wmax, layers[l]->W);
  auto mask_slot = [&](int t, int l) -> uint32_t* {
    return mask_trace == nullptr ? nullptr : mask_trace + ((size_t)t * n_layers + l) * batch * Wmax;
  };
  auto y_slot = [&](int t, int l) -> float* {
    return y_trace == nullptr ? nullptr : y_trace + ((size_t)t * n_layers + l) * batch * d0.d_model;
  };
  if (mask_trace != nullptr)  // words past a narrower layer's count stay zero
    SFFN_CUDA(cudaMemsetAsync(mask_trace, 0, (size_t)n_steps * n_layers * batch * Wmax * sizeof(uint32_t), s),
              "mask trace clear");
  // look-ahead mask words: call k reads buffer k % 2 and predicts into the other
  const size_t lab = align_up((size_t)Wmax * sizeof(uint32_t), 256);
  uint32_t* labuf[2] = {reinterpret_cast<uint32_t*>(base + per + 2 * xb + 2 * yb),
                        reinterpret_cast<uint32_t*>(base + per + 2 * xb + 2 * yb + lab)};

  bool all_fused = batch == 1;
  for (int l = 0; l < n_layers; ++l) all_fused = all_fused && layers[l]->fused();
  if (all_fused) {
    // Residual + LayerNorm is formed at the start of the next layer's kernel:
    // the kernel of (step t, layer l) reads the previous layer's input and
    // output and writes this layer's input.  A last LayerNorm launch closes
    // the final step.
    const void* xprev = nullptr;  // input of the previous layer
    const float* yprev = nullptr;  // output of the previous layer
    int k = 0;                     // running layer counter (ping-pong index)
    if (lookahead) {  // call 0's mask: the first layer's predictor on x0
      Ws ws;
      SFFN_TRY(check_ws(layers[0], batch, workspace, per, &ws));
      LookAhead la;
      la.pred = layers[0];
      la.la_out = labuf[0];
      la.predict_only = true;
      SFFN_TRY(run_layer(layers[0], x0, nullptr, nullptr, nullptr, nullptr, 0.f, nullptr, nullptr, ws, s, la));
    }
    for (int t = 0; t < n_steps; ++t) {
      for (int l = 0; l < n_layers; ++l, ++k) {
        const sffn_layer* L = layers[l];
        Ws ws;
        SFFN_TRY(check_ws(L, batch, workspace, per, &ws));
        float* ycur = y_trace != nullptr ? y_slot(t, l) : ybufs[k & 1];
        uint32_t* mcur = mask_slot(t, l);
        // look-ahead: this call's mask was predicted by the previous call; this
        // call predicts the next layer's (the last call's prediction is unused)
        LookAhead la;
        if (lookahead) {
          la.pred = layers[(l + 1) % n_layers];
          la.la_in = labuf[k & 1];
          la.la_out = labuf[(k + 1) & 1];
          mcur = nullptr;
        }
        void* xin_store;  // where this layer's input lives
        if (k == 0) {
          xin_store = const_cast<void*>(x0);
          if (trace != nullptr)
            SFFN_CUDA(cudaMemcpyAsync(trace, x0, xbytes, cudaMemcpyDeviceToDevice, s), "trace copy");
          SFFN_TRY(run_layer(L, x0, nullptr, nullptr, nullptr, nullptr, 0.f, ycur, mcur, ws, s, la));
        } else {
          if (l == 0)
            xin_store = xo + (size_t)(t - 1) * xbytes;  // last step's output is this step's input
          else if (trace != nullptr)
            xin_store = trace + ((size_t)t * n_layers + l) * xbytes;
          else
            xin_store = xbuf[k & 1];
          SFFN_TRY(run_layer(L, xprev, yprev, xin_store, ln_gamma, ln_beta, ln_eps, ycur, mcur, ws, s, la));
          if (l == 0 && trace != nullptr)
            SFFN_CUDA(cudaMemcpyAsync(trace + (size_t)t * n_layers * xbytes, xin_store, xbytes,
                                      cudaMemcpyDeviceToDevice, s),
                      "trace copy");
        }
        if (lookahead && mask_trace != nullptr)  // the mask this call used, before call k + 1 reuses the buffer
          SFFN_CUDA(cudaMemcpyAsync(mask_slot(t, l), labuf[k & 1], (size_t)L->W * sizeof(uint32_t),
                                    cudaMemcpyDeviceToDevice, s),
                    "mask trace copy");
        xprev = xin_store;
        yprev = ycur;
      }
    }
    SFFN_CUDA(launch_residual_layernorm(d0.dtype, xprev, yprev, batch, d0.d_model, ln_gamma, ln_beta, ln_eps,
                                        xo + (size_t)(n_steps - 1) * xbytes, s),
              "layernorm launch");
    return SFFN_OK;
  }

  const void* xin = x0;
  for (int t = 0; t < n_steps; ++t) {
    for (int l = 0; l < n_layers; ++l) {
      const sffn_layer* L = layers[l];
      if (trace != nullptr)
        SFFN_CUDA(cudaMemcpyAsync(trace + ((size_t)t * n_layers + l) * xbytes, xin, xbytes,
                                  cudaMemcpyDeviceToDevice, s),
                  "trace copy");
      Ws ws;
      SFFN_TRY(check_ws(L, batch, workspace, per, &ws));
      SFFN_TRY(run_predictor(L, xin, batch, ws, nullptr, s));
      if (mask_trace != nullptr)
        SFFN_CUDA(cudaMemcpy2DAsync(mask_slot(t, l), (size_t)Wmax * sizeof(uint32_t), ws.mask(),
                                    (size_t)L->W * sizeof(uint32_t), (size_t)L->W * sizeof(uint32_t), batch,
                                    cudaMemcpyDeviceToDevice, s),
                  "mask trace copy");
      float* ycur = y_trace != nullptr ? y_slot(t, l) : ybuf;
      SFFN_TRY(run_sparse_ffn(L, xin, batch, ycur, ws, s));
      void* xnext = (l == n_layers - 1) ? static_cast<void*>(xo + (size_t)t * xbytes) : xbuf[l & 1];
      SFFN_CUDA(launch_residual_layernorm(d0.dtype, xin, ycur, batch, d0.d_model, ln_gamma, ln_beta, ln_eps,
                                          xnext, s),
                "layernorm launch");
      xin = xnext;
    }
  }
  return SFFN_OK;
}

sffn_status sffn_profile_counts(sffn_layer_t L, const void* X, int32_t n_tokens, int32_t* counts, void* workspace,
                                size_t ws_bytes, void* stream) {
  g_err.clear();
  if (L == nullptr) return fail(SFFN_ERR_INVALID_ARG, "layer is NULL");
  if (n_tokens < 1) return fail(SFFN_ERR_INVALID_ARG, "n_tokens must be >= 1");
  SFFN_TRY(check_dev_ptr(X, "X"));
  if (counts == nullptr) return fail(SFFN_ERR_INVALID_ARG, "counts is NULL");
  const int chunk = std::min(L->desc.max_batch, 8);
  Ws ws;
  SFFN_TRY(check_ws(L, chunk, workspace, ws_bytes, &ws));
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  SFFN_CUDA(cudaMemsetAsync(counts, 0, (size_t)L->desc.d_ff * sizeof(int32_t), s), "counts memset");
  const unsigned char* xb = static_cast<const unsigned char*>(X);
  for (int t0 = 0; t0 < n_tokens; t0 += chunk) {
    const int nb = std::min(chunk, n_tokens - t0);
    SFFN_TRY(run_predictor(L, xb + (size_t)t0 * L->desc.d_model * L->esize, nb, ws, nullptr, s));
    SFFN_CUDA(launch_count_bits(ws.mask(), nb, L->desc.d_ff, L->W, counts, s), "count launch");
  }
  return SFFN_OK;
}

sffn_status sffn_hot_first_perm(const int32_t* counts, int32_t d_ff, int32_t* perm) {
  g_err.clear();
  if (counts == nullptr || perm == nullptr || d_ff < 1) return fail(SFFN_ERR_INVALID_ARG, "bad arguments");
  std::vector<int32_t> order(d_ff);
  std::iota(order.begin(), order.end(), 0);
  std::stable_sort(order.begin(), order.end(), [&](int32_t a, int32_t b) { return counts[a] > counts[b]; });
  std::copy(order.begin(), order.end(), perm);
  return SFFN_OK;
}

sffn_status sffn_permute_rows(const void* src, void* dst, const int32_t* perm, int32_t rows, int64_t row_bytes,
                              void* stream) {
  g_err.clear();
  if (src == nullptr || dst == nullptr || (reinterpret_cast<uintptr_t>(src) & 3) || (reinterpret_cast<uintptr_t>(dst) & 3))
    return fail(SFFN_ERR_INVALID_ARG, "src/dst NULL or not 4-byte aligned");
  if (perm == nullptr || rows < 1 || row_bytes <= 0 || row_bytes % 4 != 0)
    return fail(SFFN_ERR_INVALID_ARG, "bad perm/rows/row_bytes (row_bytes must be a multiple of 4)");
  if (src == dst) return fail(SFFN_ERR_INVALID_ARG, "permute_rows is out of place");
  SFFN_CUDA(launch_permute_rows(src, dst, perm, rows, row_bytes, static_cast<cudaStream_t>(stream)),
            "permute launch");
  return SFFN_OK;
}

sffn_status sffn_bundle_rows(const void* w_up, const void* w_gate, const void* w_downT, int32_t d_ff,
                             int32_t d_model, int32_t dtype, void* bundle, void* stream) {
  g_err.clear();
  if (dtype != SFFN_F32 && dtype != SFFN_F16 && dtype != SFFN_BF16)
    return fail(SFFN_ERR_INVALID_ARG, "unknown dtype %d", dtype);
  const size_t esize = dtype == SFFN_F32 ? 4 : 2;
  if (d_ff < 1 || d_model < 1 || ((size_t)d_model * esize) % 16 != 0)
    return fail(SFFN_ERR_INVALID_ARG, "bad d_ff/d_model (d_model * sizeof(dtype) must be a multiple of 16)");
  SFFN_TRY(check_dev_ptr(w_up, "w_up"));
  SFFN_TRY(check_dev_ptr(w_downT, "w_downT"));
  SFFN_TRY(check_dev_ptr(bundle, "bundle"));
  if (w_gate != nullptr) SFFN_TRY(check_dev_ptr(w_gate, "w_gate"));
  const size_t rb = (size_t)d_model * esize;
  const int nrows = w_gate != nullptr ? 3 : 2;
  const void* src[3] = {w_gate, w_up, w_downT};
  unsigned char* dst = static_cast<unsigned char*>(bundle);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int k = 0;
  for (int m = w_gate != nullptr ? 0 : 1; m < 3; ++m, ++k)  // matrix m's rows into column block k of the bundle
    SFFN_CUDA(cudaMemcpy2DAsync(dst + (size_t)k * rb, (size_t)nrows * rb, src[m], rb, rb, (size_t)d_ff,
                                cudaMemcpyDeviceToDevice, s),
              "bundle copy");
  return SFFN_OK;
}

sffn_status sffn_read_device_status(void* workspace, int32_t* status, void* stream) {
  g_err.clear();
  if (workspace == nullptr || status == nullptr) return fail(SFFN_ERR_INVALID_ARG, "NULL argument");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  WsHeader h;
  SFFN_CUDA(cudaMemcpyAsync(&h, workspace, sizeof(h), cudaMemcpyDeviceToHost, s), "status read");
  SFFN_CUDA(cudaStreamSynchronize(s), "status sync");
  *status = (int32_t)h.status;
  if (h.status != 0) {
    // clear the status; after a timeout the barrier words may be mid-generation
    WsHeader z;
    std::memset(&z, 0, sizeof(z));

    SFFN_CUDA(cudaMemcpyAsync(workspace, &z, sizeof(z), cudaMemcpyHostToDevice, s), "status clear");
    SFFN_CUDA(cudaStreamSynchronize(s), "status clear sync");
  }
  return SFFN_OK;
}

sffn_status sffn_debug_occupy(int64_t ns, int32_t blocks, int32_t smem_bytes, void* stream) {
  g_err.clear();
  if (ns <= 0 || ns > 2000000000LL) return fail(SFFN_ERR_INVALID_ARG, "ns outside (0, 2e9]");
  if (blocks < 1 || blocks > 65535) return fail(SFFN_ERR_INVALID_ARG, "blocks outside [1, 65535]");
  int dev = 0, optin = 0;
  SFFN_CUDA(cudaGetDevice(&dev), "device query");
  SFFN_CUDA(cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev), "device query");
  if (smem_bytes < 0 || smem_bytes > optin) return fail(SFFN_ERR_INVALID_ARG, "smem_bytes outside [0, %d]", optin);
  SFFN_CUDA(launch_occupy((uint64_t)ns, blocks, (size_t)smem_bytes, static_cast<cudaStream_t>(stream)),
            "occupy launch");
  return SFFN_OK;
}

sffn_status sffn_debug_wait_timeout(void* workspace, size_t ws_bytes, int64_t timeout_ns, void* stream) {
  g_err.clear();
  if (workspace == nullptr || ws_bytes < sizeof(WsHeader) + barrier_flag_bytes(2))
    return fail(SFFN_ERR_WORKSPACE, "workspace too small");
  if (timeout_ns <= 0 || timeout_ns > 10000000000LL) return fail(SFFN_ERR_INVALID_ARG, "timeout out of range");
  SFFN_CUDA(launch_wait_timeout(static_cast<WsHeader*>(workspace),
                                reinterpret_cast<uint32_t*>(static_cast<unsigned char*>(workspace) + sizeof(WsHeader)),
                                (uint64_t)timeout_ns,
                                static_cast<cudaStream_t>(stream)),
            "wait launch");
  return SFFN_OK;
}

}  // extern "C"

// ---- internals of sffn_forward_noalloc (noalloc.cu): the single-launch layer
// kernel on a fixed scratch array instead of a workspace.

sffn_status sffn_internal_fail(sffn_status status, const char* message) { return fail(status, "%s", message); }

sffn_status sffn_internal_layer_device(sffn_layer_t L, int* device) {
  g_err.clear();
  if (L == nullptr) return fail(SFFN_ERR_INVALID_ARG, "layer is NULL");
  *device = L->device;
  return SFFN_OK;
}

sffn_status sffn_internal_layer_on_scratch(sffn_layer_t L, const void* x, float* y, void* scratch,
                                           size_t scratch_bytes, void* stream) {
  if (!L->fused())
    return fail(SFFN_ERR_UNSUPPORTED, "the layer has no single-launch kernel configuration (or asks for the "
                                      "multi-kernel path)");
  SFFN_TRY(check_dev_ptr(x, "x"));
  SFFN_TRY(check_dev_ptr(y, "y"));
  const auto& d = L->desc;
  // header, barrier flags, the launch's h slots -- the workspace layout's order
  const size_t flags_off = align_up(sizeof(WsHeader), 256);
  const size_t part_off = flags_off + align_up(barrier_flag_bytes((uint32_t)L->layer_grid), 256);
  const size_t need = part_off + align_up(layer_slot_bytes(d.rank), 256);
  if (need > scratch_bytes)
    return fail(SFFN_ERR_UNSUPPORTED, "this layer needs %zu bytes of scratch, the fixed array holds %zu", need,
                scratch_bytes);
  unsigned char* base = static_cast<unsigned char*>(scratch);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // The launch counter, the barrier words and the slots must start at zero
  // (the array keeps whatever the last call left, possibly mid-count after a
  // timed-out wait); the status word and its detail (the header's first eight
  // bytes) are kept until sffn_noalloc_read_status reads and clears them.
  constexpr size_t kKeep = 2 * sizeof(uint32_t);
  static_assert(offsetof(WsHeader, status) == 0 && offsetof(WsHeader, detail) == 4, "status words first");
  SFFN_CUDA(cudaMemsetAsync(base + kKeep, 0, need - kKeep, s), "scratch clear");
  LayerArgs a{};
  a.x = x;
  a.V = d.pred_V;
  a.U = d.pred_U;
  a.pb = d.pred_b;
  a.b = d.b;
  a.tau = d.tau;
  a.w_up = d.w_up;
  a.w_gate = d.w_gate;
  a.w_downT = d.w_downT;
  a.y = y;
  a.h_slots = reinterpret_cast<unsigned long long*>(base + part_off);
  a.hdr = reinterpret_cast<WsHeader*>(base);
  a.bar_flags = reinterpret_cast<uint32_t*>(base + flags_off);
  a.d = d.d_model;
  a.f = d.d_ff;
  a.r = d.rank;
  a.act = d.act;
  a.nstages = L->lcfg.nstages;
  a.u_smem = L->lcfg.u_smem;
  a.region_bytes = L->lcfg.region_bytes;
  a.u_off = L->lcfg.u_off;
  a.hot_rows = d.hot_rows;
  a.warm_rows = d.warm_rows;
  a.hot_stages = L->lcfg.hot_stages;
  a.balance = 0;
  a.cluster = L->layer_cluster;
  a.static_weights = (d.flags & SFFN_FLAG_STATIC_WEIGHTS) ? 1 : 0;
  a.prefill = 0;
  a.wait_ns = (uint64_t)g_wait_ns;
  a.wstride = L->wstride;
  SFFN_CUDA(launch_layer(d.dtype, L->lcfg, a, L->layer_grid, s), "layer launch");
  return SFFN_OK;
}

