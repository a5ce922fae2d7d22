// capi.cu — the extern "C" boundary of libcsa2.so: host-side validation,
// workspace carving and the CSA2 layer-group orchestration.
//
// [CSA2] wire.sakhanda.co, "DeepSeek AI выпустила DeepSeek-V4.1-Flash ...",
//        section "Сжатое разреженное внимание 2 (CSA2)": static layer modes
//        Full / Reindex / Reuse; the Full layer forms the hierarchical pool.
// [TG]   tgviewer.app, "DeepSeek-V4.1-Flash: Frontier Agents on a Smaller
//        Memory Budget", CSA2 bullet: Reuse layers share the Top-K indices and
//        skip re-scoring.
//
// Every entry point validates its arguments on the host, enqueues its
// kernels on the caller's stream and returns a csa2_status; nothing here
// synchronises the host or allocates device memory.
#include <atomic>
#include <cstdio>
#include <mutex>

#include "common.cuh"

namespace csa2 {

// ---- kernels' host launchers (defined in the other translation units) -------
int launch_quantize_fp4(const void* x, int B, int64_t rows, const int64_t* pos, uint8_t* codes,
                        uint8_t* scales, int64_t n_cap, int32_t* st, cudaStream_t s);
int launch_append_indexer_k(const uint8_t* k_new, int B, int64_t rows, int d_I, const int64_t* pos,
                            uint8_t* kI, uint8_t* kbar, int64_t n_cap, int32_t* st, cudaStream_t s);
int launch_block_means(const uint8_t* kI, int B, int d_I, const int64_t* n, int64_t n_max,
                       int64_t n_cap, uint8_t* kbar, int32_t* st, cudaStream_t s);
int launch_append_swa(const void* x, int B, int d, const int64_t* pos, void* swa, int W,
                      cudaStream_t s);
int launch_swa_ring(const void* const* src, void* const* dst, int L, int W, int B, int d, const int64_t* n,
                    int to_ring, int32_t* swa_len_out, cudaStream_t s);
int launch_append_step(const void* kv_new, const uint8_t* kI_new, const void* const* swa_new, void* const* swa,
                       int L, int W, int B, int d_I, const int64_t* pos, int ratio, uint8_t* codes,
                       uint8_t* scales, uint8_t* kI, uint8_t* kbar, int64_t n_cap, int64_t* n_vis_out,
                       int32_t* swa_len_out, int32_t* st, cudaStream_t s);
int launch_index_scan(const uint8_t* qI, const float* w, const uint8_t* kI, int64_t kI_seq_stride, int rps,
                      const int64_t* n, int len_div, int B, int H_I, int d_I, int64_t n_max, float* scores,
                      int64_t scores_stride, const int32_t* pool, int P, int32_t* cand_pos,
                      uint32_t* hist, TopkHdr* hdr, int topk_k, int32_t* st, cudaStream_t s);
size_t topk_ws_bytes(int B);
uint32_t* topk_ws_hist(void* ws);
TopkHdr* topk_ws_hdr(void* ws, int B);
int topk_prepare(void* ws, int B, cudaStream_t s);
int launch_topk(const float* scores, const int32_t* cand_pos, int64_t stride, const int64_t* n,
                int len_div, int B, int64_t n_max, int k, int32_t* idx_out, void* ws, bool hist_ready,
                cudaStream_t s);
size_t pool_block_max_ws_bytes(int B, int64_t n_max);
int launch_pool_block_max(const float* scores, int64_t stride, const int64_t* n, int B, int64_t n_max, int P,
                          int32_t* pool_out, void* ws, cudaStream_t s);
int topk_init_attributes();
int prefill_init_attributes();
int scan_init_attributes();
int attn_tc_init_attributes();
int launch_prefill_index(const uint8_t* qI, const float* w, int Q, const uint8_t* kI, int64_t n_keys, float* scores,
                         int64_t stride, int32_t* st, cudaStream_t s);
size_t prefill_select_ws_bytes(int Q, int64_t n_keys);
int launch_prefill_candidates(const uint8_t* qI, const float* w, int Q, const uint8_t* kI, int64_t n_keys,
                              const int64_t* n_vis, void* tk, void* sel_ws, int32_t* st, cudaStream_t s);
int launch_prefill_finish(const uint8_t* qI, const float* w, int Q, const uint8_t* kI, int64_t n_keys,
                          const int64_t* n_vis, int k, int32_t* idx, float* scores, void* tk, void* sel_ws,
                          int32_t* st, cudaStream_t s);
size_t attn_ws_bytes(int64_t units, int H, int k, int W);
size_t attn_group_ws_bytes(int64_t B, int H, int k, int W);
int launch_sparse_attn(const AttnLayers& lay, int L, int B, int H, const uint8_t* codes, const uint8_t* scales,
                       int64_t kv_seq_stride, int64_t n_cap, const int32_t* idx, int k, int64_t swa_seq_stride,
                       int W, int swa_tail, int rps, const int32_t* swa_len, float softmax_scale, void* ws,
                       int32_t* st, bool early, cudaStream_t s);

static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

// The layers [l0, l0 + L) of a group as one attention launch's operands.
static bool attn_layers(AttnLayers* lay, const void* const* q, const void* const* swa, void* const* out, int l0,
                        int L) {
  *lay = AttnLayers{};
  for (int i = 0; i < L; ++i) {
    const void *qi = q[l0 + i], *si = swa[l0 + i];
    void* oi = out[l0 + i];
    if (!qi || !si || !oi || !aligned16(qi) || !aligned16(si) || !aligned16(oi)) return false;
    lay->q[i] = static_cast<const __nv_bfloat16*>(qi);
    lay->swa[i] = static_cast<const __nv_bfloat16*>(si);
    lay->out[i] = static_cast<__nv_bfloat16*>(oi);
  }
  return true;
}

// ---- bookkeeping --------------------------------------------------------------
static std::atomic<uint64_t> g_launches{0};
void count_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

// Test hook: see csa2_debug_set_fault.
static std::atomic<int> g_fault{kFaultNone};
static std::atomic<uint64_t> g_wait_ns{2000000000ull};
int debug_fault() { return g_fault.load(std::memory_order_relaxed); }
uint64_t debug_wait_ns() { return g_wait_ns.load(std::memory_order_relaxed); }
// The text of the last CUDA error a call of this thread ran into.
static thread_local char g_cuda_error[160] = "";
int launch_status() {
  const cudaError_t e = cudaGetLastError();
  if (e == cudaSuccess) return CSA2_OK;
  snprintf(g_cuda_error, sizeof(g_cuda_error), "%s: %s", cudaGetErrorName(e), cudaGetErrorString(e));
  return CSA2_ERR_CUDA;
}
void note_cuda_error(cudaError_t e) {
  if (e != cudaSuccess)
    snprintf(g_cuda_error, sizeof(g_cuda_error), "%s: %s", cudaGetErrorName(e), cudaGetErrorString(e));
}

// Kernel attributes (dynamic shared memory above 48 KB) are set once per
// device, on the first call that runs on it.
static int ensure_init() {
  static std::mutex mu;
  static uint64_t done_mask = 0;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return CSA2_ERR_CUDA;
  std::lock_guard<std::mutex> lk(mu);
  if (done_mask & (1ull << dev)) return CSA2_OK;
  int rc = topk_init_attributes();
  if (rc == CSA2_OK) rc = prefill_init_attributes();
  if (rc == CSA2_OK) rc = scan_init_attributes();
  if (rc == CSA2_OK) rc = attn_tc_init_attributes();
  if (rc == CSA2_OK) done_mask |= (1ull << dev);
  return rc;
}

static size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }
static bool ws_ok(const void* ws, size_t have, size_t need) {
  return need == 0 || (ws != nullptr && have >= need && (reinterpret_cast<uintptr_t>(ws) & 255) == 0);
}

// Workspace needs of the individual ops.
static size_t ws_index_full(int B, int64_t n_max) {
  return align256((size_t)B * (size_t)n_max * 4) + topk_ws_bytes(B);
}
static size_t ws_reindex(int B, int P) {
  const size_t slots = (size_t)B * (size_t)P * kBlock;
  return align256(slots * 4) * 2 + topk_ws_bytes(B);
}
static size_t ws_form_pool(int B, int64_t n_max) {
  const int64_t nb = (n_max + kBlock - 1) / kBlock;
  return align256((size_t)B * (size_t)nb * 4) + topk_ws_bytes(B);
}

static bool topk_k_ok(int k) { return k >= 1 && k <= kMaxTopK; }

// Records a caller's timing event; inside a stream capture it becomes an
// event-record node of the graph (external record), so replays time too.
static int rec(cudaEvent_t e, cudaStream_t s) {
  if (e == nullptr) return CSA2_OK;
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(s, &cs) != cudaSuccess) return CSA2_ERR_CUDA;
  const cudaError_t r = cs == cudaStreamCaptureStatusActive ? cudaEventRecordWithFlags(e, s, cudaEventRecordExternal)
                                                            : cudaEventRecord(e, s);
  return r == cudaSuccess ? CSA2_OK : CSA2_ERR_CUDA;
}

// Full indexer: zero the Top-K header, scan with the fused histogram, select.
// e_begin / e_end (optional) are recorded around the scan kernel alone.
static int full_indexer(const uint8_t* qI, const float* w, const uint8_t* kI, int64_t kI_seq_stride, int rps,
                        const int64_t* n, int B, int H_I, int d_I, int64_t n_max, int k, int32_t* idx_out,
                        float* scores_out, void* ws, int32_t* st, cudaStream_t s, cudaEvent_t e_begin,
                        cudaEvent_t e_end) {
  int rc;
  float* scores = scores_out ? scores_out : static_cast<float*>(ws);
  void* tk = static_cast<char*>(ws) + align256((size_t)B * (size_t)n_max * 4);
  // several query rows per sequence: the scan reads each key tile once for
  // all of them and writes plain scores; Top-K builds its own histogram
  const bool shared_scan = rps == 2 || rps == 4 || rps == 8;
  if (!shared_scan && (rc = topk_prepare(tk, B, s)) != CSA2_OK) return rc;
  if ((rc = rec(e_begin, s)) != CSA2_OK) return rc;
  if ((rc = launch_index_scan(qI, w, kI, kI_seq_stride, rps, n, 1, B, H_I, d_I, n_max, scores, n_max, nullptr, 0,
                              nullptr, shared_scan ? nullptr : topk_ws_hist(tk),
                              shared_scan ? nullptr : topk_ws_hdr(tk, B), k, st, s)) != CSA2_OK)
    return rc;
  if ((rc = rec(e_end, s)) != CSA2_OK) return rc;
  return launch_topk(scores, nullptr, n_max, n, 1, B, n_max, k, idx_out, tk, !shared_scan, s);
}

// e_begin / e_end (optional) are recorded around the block-mean scan alone.
static int pool_indexer(const uint8_t* qI, const float* w, const uint8_t* kbar, int64_t kbar_seq_stride, int rps,
                        const int64_t* n, int B, int H_I, int d_I, int64_t n_max, int P, int32_t* pool_out,
                        void* ws, int32_t* st, cudaStream_t s, cudaEvent_t e_begin = nullptr,
                        cudaEvent_t e_end = nullptr) {
  int rc;
  const int64_t nb_max = (n_max + kBlock - 1) / kBlock;     // rows of block means
  float* scores = static_cast<float*>(ws);
  void* tk = static_cast<char*>(ws) + align256((size_t)B * (size_t)nb_max * 4);
  if ((rc = topk_prepare(tk, B, s)) != CSA2_OK) return rc;
  if ((rc = rec(e_begin, s)) != CSA2_OK) return rc;
  if ((rc = launch_index_scan(qI, w, kbar, kbar_seq_stride, rps, n, kBlock, B, H_I, d_I, nb_max, scores, nb_max,
                              nullptr, 0, nullptr, topk_ws_hist(tk), topk_ws_hdr(tk, B), P, st, s)) != CSA2_OK)
    return rc;
  if ((rc = rec(e_end, s)) != CSA2_OK) return rc;
  return launch_topk(scores, nullptr, nb_max, n, kBlock, B, nb_max, P, pool_out, tk, true, s);
}

static int reindex_indexer(const uint8_t* qI, const float* w, const uint8_t* kI, int64_t kI_seq_stride, int rps,
                           const int64_t* n, const int32_t* pool, int P, int B, int H_I, int d_I, int k,
                           int32_t* idx_out, void* ws, int32_t* st, cudaStream_t s, cudaEvent_t e_begin,
                           cudaEvent_t e_end) {
  int rc;
  const int64_t slots = (int64_t)P * kBlock;
  float* scores = static_cast<float*>(ws);
  int32_t* cpos = reinterpret_cast<int32_t*>(static_cast<char*>(ws) + align256((size_t)B * slots * 4));
  void* tk = static_cast<char*>(ws) + 2 * align256((size_t)B * slots * 4);
  if ((rc = topk_prepare(tk, B, s)) != CSA2_OK) return rc;
  if ((rc = rec(e_begin, s)) != CSA2_OK) return rc;
  // The pool scan writes every one of the P*8 slots of every row (absent
  // positions carry cand_pos -1), so Top-K takes all slots of each row.
  if (P > 0 && (rc = launch_index_scan(qI, w, kI, kI_seq_stride, rps, n, 1, B, H_I, d_I, INT64_MAX, scores, slots,
                                       pool, P, cpos, topk_ws_hist(tk), topk_ws_hdr(tk, B), k, st, s)) != CSA2_OK)
    return rc;
  if ((rc = rec(e_end, s)) != CSA2_OK) return rc;
  return launch_topk(scores, cpos, slots, nullptr, 1, B, slots, k, idx_out, tk, true, s);
}
static bool index_dims_ok(int H_I, int d_I) { return H_I >= 1 && H_I <= 8 && (d_I == 64 || d_I == 128); }

}  // namespace csa2

using namespace csa2;

extern "C" {

const char* csa2_status_string(int status) {
  switch (status) {
    case CSA2_OK: return "CSA2_OK";
    case CSA2_ERR_INVALID_ARG: return "CSA2_ERR_INVALID_ARG";
    case CSA2_ERR_UNSUPPORTED_SHAPE: return "CSA2_ERR_UNSUPPORTED_SHAPE";
    case CSA2_ERR_WORKSPACE: return "CSA2_ERR_WORKSPACE";
    case CSA2_ERR_CUDA: return "CSA2_ERR_CUDA";
    case CSA2_ERR_TIMEOUT: return "CSA2_ERR_TIMEOUT";
    case CSA2_ERR_DEVICE_BOUNDS: return "CSA2_ERR_DEVICE_BOUNDS";
    case CSA2_ERR_DEVICE_RANGE: return "CSA2_ERR_DEVICE_RANGE";
    default: return "CSA2_ERR_UNKNOWN";
  }
}

int csa2_version(void) { return 102; }

uint64_t csa2_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

const char* csa2_last_cuda_error(void) { return g_cuda_error; }

int csa2_debug_set_fault(int32_t fault, int64_t wait_ns) {
  if (fault < kFaultNone || fault > kFaultPrefill || wait_ns < 0) return CSA2_ERR_INVALID_ARG;
  g_fault.store(fault, std::memory_order_relaxed);
  g_wait_ns.store(wait_ns > 0 ? (uint64_t)wait_ns : 2000000000ull, std::memory_order_relaxed);
  return CSA2_OK;
}

size_t csa2_workspace_size(int32_t op, int32_t B, int64_t n_max, int32_t k, int32_t P, int32_t H) {
  if (B < 0 || n_max < 0) return 0;
  switch (op) {
    case CSA2_OP_TOPK: return topk_ws_bytes(B);
    case CSA2_OP_INDEX_FULL: return ws_index_full(B, n_max);
    case CSA2_OP_INDEX_REINDEX: return ws_reindex(B, P);
    case CSA2_OP_FORM_POOL: return ws_form_pool(B, n_max);
    case CSA2_OP_SPARSE_ATTN: return attn_ws_bytes(B, H, k, 128);
    case CSA2_OP_PREFILL_GROUP: {
      // B = queries, n_max = entries: full score rows (written only for the
      // query tiles whose candidates cannot serve them) + Top-K + attention
      // partials + the sampled scores, thresholds and tile marks
      size_t m = align256((size_t)B * (size_t)n_max * 4) + topk_ws_bytes(B);
      return m + align256(attn_group_ws_bytes(B, H, k, 128)) + prefill_select_ws_bytes(B, n_max);
    }
    case CSA2_OP_FORM_POOL_BLOCK_MAX: return pool_block_max_ws_bytes(B, n_max);
    case CSA2_OP_LAYER_GROUP: {
      // the block-max pool reads the Full scores, so its workspace follows them
      size_t m = ws_index_full(B, n_max) + pool_block_max_ws_bytes(B, n_max);
      const size_t r = ws_reindex(B, P), f = ws_form_pool(B, n_max), a = attn_group_ws_bytes(B, H, k, 128);
      if (r > m) m = r;
      if (f > m) m = f;
      if (a > m) m = a;
      return m;
    }
    default: return 0;
  }
}

int csa2_quantize_kv_fp4(const void* x, int32_t B, int64_t rows, int32_t d, const int64_t* pos,
                         uint8_t* codes, uint8_t* scales, int64_t n_cap, int32_t* d_status,
                         void* stream) {
  if (B < 0 || rows < 0 || n_cap < 0) return CSA2_ERR_INVALID_ARG;
  if (d != 512) return CSA2_ERR_UNSUPPORTED_SHAPE;
  if ((int64_t)B * rows == 0) return CSA2_OK;
  if (!x || !codes || !scales || !aligned16(x) || !aligned16(codes) || !aligned16(scales))
    return CSA2_ERR_INVALID_ARG;
  return launch_quantize_fp4(x, B, rows, pos, codes, scales, n_cap, d_status,
                             static_cast<cudaStream_t>(stream));
}

int csa2_append_indexer_k(const uint8_t* k_new, int32_t B, int64_t rows, int32_t d_I,
                          const int64_t* pos, uint8_t* kI, uint8_t* kbar, int64_t n_cap,
                          int32_t* d_status, void* stream) {
  if (B < 0 || rows < 0 || n_cap < 0) return CSA2_ERR_INVALID_ARG;
  if (d_I != 64 && d_I != 128) return CSA2_ERR_UNSUPPORTED_SHAPE;
  if ((int64_t)B * rows == 0) return CSA2_OK;
  if (!k_new || !kI || !aligned16(k_new) || !aligned16(kI) || (kbar && !aligned16(kbar)))
    return CSA2_ERR_INVALID_ARG;
  return launch_append_indexer_k(k_new, B, rows, d_I, pos, kI, kbar, n_cap, d_status,
                                 static_cast<cudaStream_t>(stream));
}

int csa2_block_means(const uint8_t* kI, int32_t B, int32_t d_I, const int64_t* n, int64_t n_max,
                     int64_t n_cap, uint8_t* kbar, int32_t* d_status, void* stream) {
  if (B < 0 || n_max < 0 || n_max > n_cap) return CSA2_ERR_INVALID_ARG;
  if (d_I != 64 && d_I != 128) return CSA2_ERR_UNSUPPORTED_SHAPE;
  if (B == 0 || n_max == 0) return CSA2_OK;
  if (!kI || !kbar || !n || !aligned16(kI) || !aligned16(kbar)) return CSA2_ERR_INVALID_ARG;
  return launch_block_means(kI, B, d_I, n, n_max, n_cap, kbar, d_status,
                            static_cast<cudaStream_t>(stream));
}

int csa2_append_swa(const void* x, int32_t B, int32_t d, const int64_t* pos, void* swa, int32_t W,
                    void* stream) {
  if (B < 0 || W <= 0) return CSA2_ERR_INVALID_ARG;
  if (d != 512) return CSA2_ERR_UNSUPPORTED_SHAPE;
  if (B == 0) return CSA2_OK;
  if (!x || !pos || !swa || !aligned16(x) || !aligned16(swa)) return CSA2_ERR_INVALID_ARG;
  return launch_append_swa(x, B, d, pos, swa, W, static_cast<cudaStream_t>(stream));
}

int csa2_append_step(const void* kv_new, const uint8_t* kI_new, const void* const* swa_new, void* const* swa,
                     int32_t L, int32_t W, int32_t B, int32_t d, int32_t d_I, const int64_t* pos,
                     uint8_t* codes, uint8_t* scales, uint8_t* kI, uint8_t* kbar, int64_t n_cap,
                     int32_t* d_status, void* stream) {
  return csa2_append_step_ratio(kv_new, kI_new, swa_new, swa, L, W, B, d, d_I, pos, 1, codes, scales, kI, kbar,
                                n_cap, nullptr, nullptr, d_status, stream);
}

int csa2_append_step_ratio(const void* kv_new, const uint8_t* kI_new, const void* const* swa_new,
                           void* const* swa, int32_t L, int32_t W, int32_t B, int32_t d, int32_t d_I,
                           const int64_t* pos, int32_t ratio, uint8_t* codes, uint8_t* scales, uint8_t* kI,
                           uint8_t* kbar, int64_t n_cap, int64_t* n_vis_out, int32_t* swa_len_out,
                           int32_t* d_status, void* stream) {
  if (B < 0 || L < 0 || n_cap < 0 || (L > 0 && W <= 0) || ratio < 1) return CSA2_ERR_INVALID_ARG;
  if (d != 512 || (d_I != 64 && d_I != 128) || L > 64) return CSA2_ERR_UNSUPPORTED_SHAPE;
  if (B == 0) return CSA2_OK;
  if (!kv_new || !kI_new || !pos || !codes || !scales || !kI || (L > 0 && (!swa_new || !swa)))
    return CSA2_ERR_INVALID_ARG;
  if (!aligned16(kv_new) || !aligned16(codes) || !aligned16(scales) || ((uintptr_t)kI_new & 3) ||
      ((uintptr_t)kI & 15) || (kbar && ((uintptr_t)kbar & 15)))
    return CSA2_ERR_INVALID_ARG;
  for (int l = 0; l < L; ++l)
    if (!swa_new[l] || !swa[l] || !aligned16(swa_new[l]) || !aligned16(swa[l])) return CSA2_ERR_INVALID_ARG;
  if (swa_len_out && W <= 0) return CSA2_ERR_INVALID_ARG;
  return launch_append_step(kv_new, kI_new, swa_new, swa, L, W, B, d_I, pos, ratio, codes, scales, kI, kbar, n_cap,
                            n_vis_out, swa_len_out, d_status, static_cast<cudaStream_t>(stream));
}

static int swa_ring_args(const void* const* a, const void* const* b, int32_t L, int32_t W, int32_t B, int32_t d,
                         const int64_t* n) {
  if (L < 0 || W <= 0 || B < 0) return CSA2_ERR_INVALID_ARG;
  if (d != 512 || L > 64) return CSA2_ERR_UNSUPPORTED_SHAPE;
  if (L > 0 && B > 0 && (!a || !b || !n)) return CSA2_ERR_INVALID_ARG;
  for (int l = 0; l < L && B > 0; ++l)
    if (!a[l] || !b[l] || !aligned16(a[l]) || !aligned16(b[l])) return CSA2_ERR_INVALID_ARG;
  return CSA2_OK;
}

int csa2_swa_export(const void* const* rings, int32_t L, int32_t W, int32_t B, int32_t d, const int64_t* n,
                    void* const* rows_out, void* stream) {
  const int rc = swa_ring_args(rings, rows_out, L, W, B, d, n);
  if (rc != CSA2_OK || L == 0 || B == 0) return rc;
  return launch_swa_ring(rings, rows_out, L, W, B, d, n, 0, nullptr, static_cast<cudaStream_t>(stream));
}

int csa2_swa_restore(const void* const* rows, int32_t L, int32_t W, int32_t B, int32_t d, const int64_t* n,
                     void* const* rings, int32_t* swa_len_out, void* stream) {
  const int rc = swa_ring_args(rows, rings, L, W, B, d, n);
  if (rc != CSA2_OK || L == 0 || B == 0) return rc;
  return launch_swa_ring(rows, rings, L, W, B, d, n, 1, swa_len_out, static_cast<cudaStream_t>(stream));
}

int csa2_index_scores(const uint8_t* qI, const float* w, const uint8_t* kI, int64_t kI_seq_stride,
                      const int64_t* n, int32_t B, int32_t H_I, int32_t d_I, int64_t n_max,
                      float* scores, int64_t scores_stride, int32_t* d_status, void* stream) {
  if (B < 0 || n_max < 0 || kI_seq_stride < 0 || scores_stride < n_max) return CSA2_ERR_INVALID_ARG;
  if (!index_dims_ok(H_I, d_I)) return CSA2_ERR_UNSUPPORTED_SHAPE;
  if (B == 0 || n_max == 0) return CSA2_OK;
  if (!qI || !w || !kI || !n || !scores || !aligned16(qI) || !aligned16(kI)) return CSA2_ERR_INVALID_ARG;
  const int rc = ensure_init();
  if (rc != CSA2_OK) return rc;
  return launch_index_scan(qI, w, kI, kI_seq_stride, 1, n, 1, B, H_I, d_I, n_max, scores, scores_stride,
                           nullptr, 0, nullptr, nullptr, nullptr, 0, d_status, static_cast<cudaStream_t>(stream));
}

int csa2_topk(const float* scores, const int32_t* cand_pos, int64_t scores_stride, const int64_t* n,
              int32_t B, int64_t n_max, int32_t k, int32_t* idx_out, void* ws, size_t ws_bytes,
              void* stream) {
  if (B < 0 || n_max < 0 || scores_stride < n_max) return CSA2_ERR_INVALID_ARG;
  if (!topk_k_ok(k) || n_max > 0x7FFFFFFF) return CSA2_ERR_UNSUPPORTED_SHAPE;
  if (B == 0) return CSA2_OK;
  if (!scores || !idx_out) return CSA2_ERR_INVALID_ARG;
  if (!ws_ok(ws, ws_bytes, topk_ws_bytes(B))) return CSA2_ERR_WORKSPACE;
  int rc = ensure_init();
  if (rc != CSA2_OK) return rc;
  return launch_topk(scores, cand_pos, scores_stride, n, 1, B, n_max, k, idx_out, ws, false,
                     static_cast<cudaStream_t>(stream));
}

int csa2_index_full(const uint8_t* qI, const float* w, const uint8_t* kI, int64_t kI_seq_stride,
                    const int64_t* n, int32_t B, int32_t H_I, int32_t d_I, int64_t n_max, int32_t k,
                    int32_t* idx_out, float* scores_out, void* ws, size_t ws_bytes,
                    int32_t* d_status, void* stream) {
  if (B < 0 || n_max < 0 || kI_seq_stride < 0) return CSA2_ERR_INVALID_ARG;
  if (!index_dims_ok(H_I, d_I) || !topk_k_ok(k) || n_max > 0x7FFFFFFF) return CSA2_ERR_UNSUPPORTED_SHAPE;
  if (B == 0) return CSA2_OK;
  if (!qI || !w || !kI || !n || !idx_out || !aligned16(qI) || !aligned16(kI)) return CSA2_ERR_INVALID_ARG;
  if (!ws_ok(ws, ws_bytes, ws_index_full(B, n_max))) return CSA2_ERR_WORKSPACE;
  int rc = ensure_init();
  if (rc != CSA2_OK) return rc;
  return full_indexer(qI, w, kI, kI_seq_stride, 1, n, B, H_I, d_I, n_max, k, idx_out, scores_out, ws, d_status,
                      static_cast<cudaStream_t>(stream), nullptr, nullptr);
}

int csa2_form_pool(const uint8_t* qI, const float* w, const uint8_t* kbar, int64_t kbar_seq_stride,
                   const int64_t* n, int32_t B, int32_t H_I, int32_t d_I, int64_t n_max, int32_t P,
                   int32_t* pool_out, void* ws, size_t ws_bytes, int32_t* d_status, void* stream) {
  if (B < 0 || n_max < 0 || kbar_seq_stride < 0) return CSA2_ERR_INVALID_ARG;
  if (!index_dims_ok(H_I, d_I) || !topk_k_ok(P) || n_max > 0x7FFFFFFF) return CSA2_ERR_UNSUPPORTED_SHAPE;
  if (B == 0) return CSA2_OK;
  if (!qI || !w || !kbar || !n || !pool_out || !aligned16(qI) || !aligned16(kbar)) return CSA2_ERR_INVALID_ARG;
  if (!ws_ok(ws, ws_bytes, ws_form_pool(B, n_max))) return CSA2_ERR_WORKSPACE;
  int rc = ensure_init();
  if (rc != CSA2_OK) return rc;
  return pool_indexer(qI, w, kbar, kbar_seq_stride, 1, n, B, H_I, d_I, n_max, P, pool_out, ws, d_status,
                      static_cast<cudaStream_t>(stream));
}

int csa2_form_pool_block_max(const float* scores, int64_t scores_stride, const int64_t* n, int32_t B,
                             int64_t n_max, int32_t P, int32_t* pool_out, void* ws, size_t ws_bytes, void* stream) {
  if (B < 0 || n_max < 0 || scores_stride < n_max) return CSA2_ERR_INVALID_ARG;
  if (!topk_k_ok(P) || n_max > 0x7FFFFFFF) return CSA2_ERR_UNSUPPORTED_SHAPE;
  if (B == 0) return CSA2_OK;
  if (!scores || !pool_out) return CSA2_ERR_INVALID_ARG;
  if (!ws_ok(ws, ws_bytes, pool_block_max_ws_bytes(B, n_max))) return CSA2_ERR_WORKSPACE;
  int rc = ensure_init();
  if (rc != CSA2_OK) return rc;
  return launch_pool_block_max(scores, scores_stride, n, B, n_max, P, pool_out, ws, static_cast<cudaStream_t>(stream));
}

int csa2_index_reindex(const uint8_t* qI, const float* w, const uint8_t* kI, int64_t kI_seq_stride,
                       const int64_t* n, const int32_t* pool, int32_t P, int32_t B, int32_t H_I,
                       int32_t d_I, int32_t k, int32_t* idx_out, void* ws, size_t ws_bytes,
                       int32_t* d_status, void* stream) {
  if (B < 0 || P < 0 || kI_seq_stride < 0) return CSA2_ERR_INVALID_ARG;
  if (!index_dims_ok(H_I, d_I) || !topk_k_ok(k) || P > kMaxTopK) return CSA2_ERR_UNSUPPORTED_SHAPE;
  if (B == 0) return CSA2_OK;
  if (!qI || !w || !kI || !n || !pool || !idx_out || !aligned16(qI) || !aligned16(kI)) return CSA2_ERR_INVALID_ARG;
  if (!ws_ok(ws, ws_bytes, ws_reindex(B, P))) return CSA2_ERR_WORKSPACE;
  int rc = ensure_init();
  if (rc != CSA2_OK) return rc;
  return reindex_indexer(qI, w, kI, kI_seq_stride, 1, n, pool, P, B, H_I, d_I, k, idx_out, ws, d_status,
                         static_cast<cudaStream_t>(stream), nullptr, nullptr);
}

int csa2_sparse_attn(const void* q, int32_t B, int32_t H, int32_t d, const uint8_t* codes,
                     const uint8_t* scales, int64_t kv_seq_stride, int64_t n_cap, const int32_t* idx,
                     int32_t k, const void* swa, int64_t swa_seq_stride, int32_t W, int32_t swa_tail,
                     const int32_t* swa_len, float softmax_scale, void* out, void* ws, size_t ws_bytes,
                     int32_t* d_status, void* stream) {
  if (B < 0 || k < 0 || W < 0 || kv_seq_stride < 0 || swa_seq_stride < 0 || n_cap < 0) return CSA2_ERR_INVALID_ARG;
  if (d != 512 || (H != 16 && H != 32 && H != 48 && H != 64) || W > 128 || k > 4096)
    return CSA2_ERR_UNSUPPORTED_SHAPE;
  if (B == 0) return CSA2_OK;
  if (!q || !out || !swa_len || (k > 0 && (!codes || !scales || !idx)) || (W > 0 && !swa))
    return CSA2_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(out) || (codes && !aligned16(codes)) || (scales && !aligned16(scales)) ||
      (swa && !aligned16(swa)))
    return CSA2_ERR_INVALID_ARG;
  if (!ws_ok(ws, ws_bytes, attn_ws_bytes(B, H, k, W))) return CSA2_ERR_WORKSPACE;
  int rc = ensure_init();
  if (rc != CSA2_OK) return rc;
  AttnLayers lay{};
  lay.q[0] = static_cast<const __nv_bfloat16*>(q);
  lay.swa[0] = static_cast<const __nv_bfloat16*>(swa);
  lay.out[0] = static_cast<__nv_bfloat16*>(out);
  return launch_sparse_attn(lay, 1, B, H, codes, scales, kv_seq_stride, n_cap, idx, k, swa_seq_stride, W,
                            swa_tail != 0, 1, swa_len, softmax_scale, ws, d_status, false,
                            static_cast<cudaStream_t>(stream));
}

static cudaEvent_t group_event(const csa2_group_args* a, int i) {
  if (a->events == nullptr || i >= a->n_events) return nullptr;
  return static_cast<cudaEvent_t>(a->events[i]);
}

int csa2_layer_group(const csa2_group_args* a, void* stream) {
  if (!a) return CSA2_ERR_INVALID_ARG;
  if (a->mode != CSA2_MODE_FULL && a->mode != CSA2_MODE_REINDEX) return CSA2_ERR_INVALID_ARG;
  if (a->n_reuse < 0 || !a->q_layers || !a->swa_layers || !a->out_layers || !a->idx) return CSA2_ERR_INVALID_ARG;
  if (a->B < 0 || a->n_max < 0 || a->n_max > a->n_cap || a->n_max > 0x7FFFFFFF) return CSA2_ERR_INVALID_ARG;
  if (a->B == 0) return CSA2_OK;
  if (!a->n || !a->codes || !a->scales || !a->kI || !a->qI || !a->w || !a->swa_len) return CSA2_ERR_INVALID_ARG;
  if (a->form_pool < CSA2_POOL_NONE || a->form_pool > CSA2_POOL_BLOCK_MAX) return CSA2_ERR_INVALID_ARG;
  if (a->rows_per_seq < 0 || a->rows_per_seq > 64 || (a->rows_per_seq > 1 && a->B % a->rows_per_seq != 0))
    return CSA2_ERR_INVALID_ARG;
  if (a->form_pool == CSA2_POOL_BLOCK_MAX && a->mode != CSA2_MODE_FULL) return CSA2_ERR_INVALID_ARG;
  if ((a->form_pool || a->mode == CSA2_MODE_REINDEX) && !a->pool) return CSA2_ERR_INVALID_ARG;
  if (a->form_pool == CSA2_POOL_MEAN_KEY && !a->kbar) return CSA2_ERR_INVALID_ARG;
  if (!index_dims_ok(a->H_I, a->d_I) || !topk_k_ok(a->k) || a->P < 0 || a->P > kMaxTopK ||
      (a->form_pool && a->P < 1) || a->d != 512 || a->W < 0 || a->W > 128 ||
      (a->H != 16 && a->H != 32 && a->H != 48 && a->H != 64))
    return CSA2_ERR_UNSUPPORTED_SHAPE;
  if (!aligned16(a->qI) || !aligned16(a->kI) || (a->kbar && !aligned16(a->kbar))) return CSA2_ERR_INVALID_ARG;
  const size_t need = csa2_workspace_size(CSA2_OP_LAYER_GROUP, a->B, a->n_cap, a->k, a->P, a->H);
  if (!ws_ok(a->ws, a->ws_bytes, need)) return CSA2_ERR_WORKSPACE;
  int rc = ensure_init();
  if (rc != CSA2_OK) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int64_t nbc = (a->n_cap + kBlock - 1) / kBlock;
  const int rps = a->rows_per_seq > 1 ? a->rows_per_seq : 1;
  const uint8_t* qp = a->qI_pool ? a->qI_pool : a->qI;
  const float* wp = a->w_pool ? a->w_pool : a->w;
  // events: [0] indexer scan begins, [1] scan ends, [2] Top-K (and pool) done,
  // [3 + l] attention of layer l done
  if (a->mode == CSA2_MODE_FULL) {
    rc = full_indexer(a->qI, a->w, a->kI, a->n_cap, rps, a->n, a->B, a->H_I, a->d_I, a->n_max, a->k, a->idx, nullptr,
                      a->ws, a->d_status, s, group_event(a, 0), group_event(a, 1));
    if (rc == CSA2_OK && a->form_pool == CSA2_POOL_MEAN_KEY)
      rc = pool_indexer(qp, wp, a->kbar, nbc, rps, a->n, a->B, a->H_I, a->d_I, a->n_max, a->P, a->pool, a->ws,
                        a->d_status, s);
    if (rc == CSA2_OK && a->form_pool == CSA2_POOL_BLOCK_MAX)   // the Full scores are still at ws
      rc = launch_pool_block_max(static_cast<const float*>(a->ws), a->n_max, a->n, a->B, a->n_max, a->P, a->pool,
                                 static_cast<char*>(a->ws) + ws_index_full(a->B, a->n_max), s);
  } else {
    // a Reindex group that forms the pool: events [0] / [1] bracket the
    // block-mean scan (its largest kernel); otherwise the Reindex scan
    if (a->form_pool)
      rc = pool_indexer(qp, wp, a->kbar, nbc, rps, a->n, a->B, a->H_I, a->d_I, a->n_max, a->P, a->pool, a->ws,
                        a->d_status, s, group_event(a, 0), group_event(a, 1));
    if (rc == CSA2_OK)
      rc = reindex_indexer(a->qI, a->w, a->kI, a->n_cap, rps, a->n, a->pool, a->P, a->B, a->H_I, a->d_I, a->k,
                           a->idx, a->ws, a->d_status, s, a->form_pool ? nullptr : group_event(a, 0),
                           a->form_pool ? nullptr : group_event(a, 1));
  }
  if (rc != CSA2_OK) return rc;
  if ((rc = rec(group_event(a, 2), s)) != CSA2_OK) return rc;
  // the group's layers share the indices and the main KV: up to
  // kMaxAttnLayers of them are attended by one launch (one CTA per row, layer
  // and key split), so their set-up, tiles and epilogues overlap
  const int n_layers = a->n_reuse + 1;
  for (int l0 = 0; l0 < n_layers; l0 += kMaxAttnLayers) {
    const int L = n_layers - l0 < kMaxAttnLayers ? n_layers - l0 : kMaxAttnLayers;
    AttnLayers lay;
    if (!attn_layers(&lay, a->q_layers, a->swa_layers, a->out_layers, l0, L)) return CSA2_ERR_INVALID_ARG;
    // one row per sequence: the layer's SWA ring (W rows, present keys first);
    // rps rows per sequence: W + rps - 1 linear rows, each window ending at its token
    // early: the call began with ordinary launches (the workspace zeroing or
    // the scan), and its later kernels write only the indices and the workspace
    rc = launch_sparse_attn(lay, L, a->B, a->H, a->codes, a->scales, a->n_cap, a->n_cap, a->idx, a->k,
                            rps > 1 ? a->W + rps - 1 : a->W, a->W, rps > 1 ? 1 : 0, rps, a->swa_len,
                            a->softmax_scale, a->ws, a->d_status, true, s);
    if (rc != CSA2_OK) return rc;
    // event 3 + l marks the end of the launch that holds layer l
    for (int l = l0; l < l0 + L; ++l)
      if ((rc = rec(group_event(a, 3 + l), s)) != CSA2_OK) return rc;
  }
  return CSA2_OK;
}

int csa2_prefill_index_scores(const uint8_t* qI, const float* w, int32_t Q, int32_t H_I, int32_t d_I,
                              const uint8_t* kI, int64_t n_keys, float* scores, int64_t scores_stride,
                              int32_t* d_status, void* stream) {
  if (Q < 0 || n_keys < 0 || scores_stride < n_keys) return CSA2_ERR_INVALID_ARG;
  if (H_I != 8 || d_I != 128 || n_keys > kMaxPrefillKeys || (int64_t)Q * 8 > 0x7FFFFFFF)
    return CSA2_ERR_UNSUPPORTED_SHAPE;
  if (Q == 0 || n_keys == 0) return CSA2_OK;
  if (!qI || !w || !kI || !scores || !aligned16(qI) || !aligned16(kI)) return CSA2_ERR_INVALID_ARG;
  int rc = ensure_init();
  if (rc != CSA2_OK) return rc;
  return launch_prefill_index(qI, w, Q, kI, n_keys, scores, scores_stride, d_status,
                              static_cast<cudaStream_t>(stream));
}

int csa2_prefill_group(const csa2_prefill_args* a, void* stream) {
  if (!a) return CSA2_ERR_INVALID_ARG;
  if (a->Q < 0 || a->n_reuse < 0 || a->n_keys < 0 || !a->q_layers || !a->swa_layers || !a->out_layers)
    return CSA2_ERR_INVALID_ARG;
  if (a->H_I != 8 || a->d_I != 128 || a->d != 512 || !topk_k_ok(a->k) || a->W < 0 || a->W > 128 ||
      (a->H != 16 && a->H != 32 && a->H != 48 && a->H != 64) || a->n_keys > kMaxPrefillKeys ||
      (int64_t)a->Q * 8 > 0x7FFFFFFF)
    return CSA2_ERR_UNSUPPORTED_SHAPE;
  if (a->Q == 0) return CSA2_OK;
  if (!a->n_vis || !a->codes || !a->scales || !a->kI || !a->qI || !a->w || !a->idx || !a->swa_len)
    return CSA2_ERR_INVALID_ARG;
  const size_t need = csa2_workspace_size(CSA2_OP_PREFILL_GROUP, a->Q, a->n_keys, a->k, 0, a->H);
  if (!ws_ok(a->ws, a->ws_bytes, need)) return CSA2_ERR_WORKSPACE;
  int rc = ensure_init();
  if (rc != CSA2_OK) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  auto ev = [&](int i) -> cudaEvent_t {
    return (a->events && i < a->n_events) ? static_cast<cudaEvent_t>(a->events[i]) : nullptr;
  };
  float* scores = static_cast<float*>(a->ws);
  void* tk = static_cast<char*>(a->ws) + align256((size_t)a->Q * (size_t)a->n_keys * 4);
  void* aws = static_cast<char*>(tk) + topk_ws_bytes(a->Q);
  void* sel = static_cast<char*>(aws) + align256(attn_group_ws_bytes(a->Q, a->H, a->k, 128));
  // events: [0] before the indexer GEMM, [1] after it (the sampled pass, the
  // thresholds and the candidate-emitting pass), [2] after Top-K, [3 + l] after layer l
  if ((rc = rec(ev(0), s)) != CSA2_OK) return rc;
  if ((rc = launch_prefill_candidates(a->qI, a->w, a->Q, a->kI, a->n_keys, a->n_vis, tk, sel, a->d_status, s)) !=
      CSA2_OK)
    return rc;
  if ((rc = rec(ev(1), s)) != CSA2_OK) return rc;
  if ((rc = launch_prefill_finish(a->qI, a->w, a->Q, a->kI, a->n_keys, a->n_vis, a->k, a->idx, scores, tk, sel,
                                  a->d_status, s)) != CSA2_OK)
    return rc;
  if ((rc = rec(ev(2), s)) != CSA2_OK) return rc;
  const int n_layers = a->n_reuse + 1;
  for (int l0 = 0; l0 < n_layers; l0 += kMaxAttnLayers) {
    const int L = n_layers - l0 < kMaxAttnLayers ? n_layers - l0 : kMaxAttnLayers;
    AttnLayers lay;
    if (!attn_layers(&lay, a->q_layers, a->swa_layers, a->out_layers, l0, L)) return CSA2_ERR_INVALID_ARG;
    // not early: the selection kernels before it are ordinary launches, so
    // the attention starts only after they end, and an early launch would
    // only move its index reads behind the window tiles
    rc = launch_sparse_attn(lay, L, a->Q, a->H, a->codes, a->scales, 0, a->n_keys, a->idx, a->k, 1, a->W, 1, 1,
                            a->swa_len, a->softmax_scale, aws, a->d_status, false, s);
    if (rc != CSA2_OK) return rc;
    for (int l = l0; l < l0 + L; ++l)
      if ((rc = rec(ev(3 + l), s)) != CSA2_OK) return rc;
  }
  return CSA2_OK;
}

}  // extern "C"
