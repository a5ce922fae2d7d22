// topk_noalloc.cu — csa2_topk_noalloc: Top-K selection that needs no
// caller-provided workspace.
//
// Some callers cannot hand the library a scratch buffer: code that runs
// inside another runtime's execution hook where device allocation is not
// allowed (an inference-engine plugin's enqueue callback, for example), code
// whose steady state must never call cudaMalloc because that call can
// synchronise the device and stall every other stream, and callers that have
// no allocator of their own at all (a plain C program driving the library
// through the C ABI). For them this entry point keeps its scratch in a
// file-scope device array that is part of the library image: it is reserved
// once per GPU when the library's device code is loaded on that GPU and held
// until the process exits. Nothing is allocated per call.
//
// The array holds the scratch of csa2_topk for at most
// CSA2_TOPK_NOALLOC_MAX_ROWS rows: 7,341,056 bytes (7.0 MiB), exactly the
// workspace csa2_topk needs for that many rows. All calls share it and it
// keeps whatever the last call left there; each call clears the part that
// must start at zero (the histograms and row headers) before use. Calls that
// overlap on the GPU — on two streams, or from two host threads without
// ordering — race on the array and give wrong results.
#include <mutex>

#include "common.cuh"

namespace csa2 {

size_t topk_ws_bytes(int B);
int topk_init_attributes();
int launch_topk(const float* scores, const int32_t* cand_pos, int64_t stride, const int64_t* n,
                int len_div, int B, int64_t n_max, int k, int32_t* idx_out, void* ws, bool hist_ready,
                cudaStream_t s);

// Scratch of csa2_topk for CSA2_TOPK_NOALLOC_MAX_ROWS rows:
//   histograms 64 x 4096 x 4 B + row headers 64 x 16 B + candidates 64 x 8192 x 8 B
//   + chunk tables 64 x 4096 x 8 B,
// each region rounded up to 256 bytes (the layout csa2_topk uses).
constexpr size_t kNoAllocScratchBytes = 1048576 + 1024 + 4194304 + 2097152;
static __device__ __align__(256) unsigned char g_topk_scratch[kNoAllocScratchBytes];

// Device address of g_topk_scratch on each device, looked up once per device
// (with that device current) on the first call made while it is current.
static void* scratch_address() {
  static std::mutex mu;
  static void* addr[64] = {nullptr};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lk(mu);
  if (addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_topk_scratch) != cudaSuccess) return nullptr;
    if (topk_init_attributes() != CSA2_OK) return nullptr;
    addr[dev] = p;
  }
  return addr[dev];
}

}  // namespace csa2

extern "C" int csa2_topk_noalloc(const float* scores, const int32_t* cand_pos, int64_t scores_stride,
                                 const int64_t* n, int32_t B, int64_t n_max, int32_t k, int32_t* idx_out,
                                 void* stream) {
  using namespace csa2;
  if (B < 0 || n_max < 0 || scores_stride < n_max) return CSA2_ERR_INVALID_ARG;
  if (k < 1 || k > kMaxTopK || n_max > 0x7FFFFFFF) return CSA2_ERR_UNSUPPORTED_SHAPE;
  if (B > CSA2_TOPK_NOALLOC_MAX_ROWS) return CSA2_ERR_UNSUPPORTED_SHAPE;
  if (topk_ws_bytes(B) > kNoAllocScratchBytes) return CSA2_ERR_UNSUPPORTED_SHAPE;
  if (B == 0) return CSA2_OK;
  if (!scores || !idx_out) return CSA2_ERR_INVALID_ARG;
  void* ws = scratch_address();
  if (ws == nullptr) return CSA2_ERR_CUDA;
  return launch_topk(scores, cand_pos, scores_stride, n, 1, B, n_max, k, idx_out, ws, false,
                     static_cast<cudaStream_t>(stream));
}
