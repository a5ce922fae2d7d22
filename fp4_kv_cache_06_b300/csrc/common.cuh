// common.cuh — shared device helpers of libcsa2 (sm_103a).
//
// PTX wrappers for the conversions and tensor-core instructions the kernels
// use, the order-preserving float key used by Top-K, and the host-side
// launch bookkeeping. Nothing here is shared with the CPU oracle.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include <utility>

#include "../../include/csa2.h"

namespace csa2 {

constexpr int kSMs = 148;              // B300: 2 dies x 74 SMs
constexpr int kMaxAttnLayers = 8;      // layers of one group attended by one launch

// Per-layer operands of one attention launch (layer = blockIdx.z). The layers
// share the Top-K indices and the FP4 main KV; each has its own queries
// [B][H][512], SWA rows and output [B][H][512].
struct AttnLayers {
  const __nv_bfloat16* q[kMaxAttnLayers];
  const __nv_bfloat16* swa[kMaxAttnLayers];
  __nv_bfloat16* out[kMaxAttnLayers];
};
constexpr int kHistBins = 4096;        // level-0 Top-K histogram (12 key bits)
constexpr int kCandCap = 8192;         // Top-K candidate buffer per row
constexpr int kMaxTopK = 2048;
constexpr int kBlock = 8;              // positions per pool block
// Prefill entries: an entry index plus a tile's 127 lanes stays below 2^31.
constexpr int64_t kMaxPrefillKeys = 0x7FFFFFFFll - 128;

// ---- host bookkeeping ------------------------------------------------------
void count_launch();
// Test hook (csa2_debug_set_fault): a kernel that must never be signalled
// once, and the bound of every device wait in nanoseconds.
constexpr int kFaultNone = 0, kFaultAttn = 1, kFaultScan = 2, kFaultPrefill = 3;
int debug_fault();
uint64_t debug_wait_ns();
int launch_status();                   // CSA2_OK or CSA2_ERR_CUDA after a launch
// After a launch that returned `e`: also clears the runtime's last error.
void note_cuda_error(cudaError_t e);    // keep the text of e for csa2_last_cuda_error
inline int launch_status(cudaError_t e) {
  const int st = launch_status();
  if (e != cudaSuccess) note_cuda_error(e);
  return e == cudaSuccess ? st : CSA2_ERR_CUDA;
}

// ---- programmatic dependent launch -----------------------------------------
// The kernels of a step are launched with programmatic stream serialization,
// so a kernel's launch and its prologue overlap the tail of the kernel before
// it. Every kernel launched this way executes pdl_wait() before its first
// global-memory access and before any return: the wait blocks until the
// preceding kernel has completed and its writes are visible (and, since that
// kernel waited in turn, everything before it), so the stream order holds.
// Without the launch attribute the wait returns at once. pdl_trigger() lets
// the next kernel start launching once every CTA of this one has issued it
// or exited; kernels that allocate TMEM issue it only after their allocation
// and allocate only after their wait, so a waiting CTA never holds columns
// that a running one still needs.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                              Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// ---- device status ---------------------------------------------------------
__device__ __forceinline__ void report(int32_t* st, int code) {
  if (st) atomicCAS(st, 0, code);
}

// ---- order-preserving key of an fp32 score (larger score -> larger key) ----
__device__ __forceinline__ uint32_t score_key(float s) {
  uint32_t u = __float_as_uint(s);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
// 64-bit composite: score desc, then position asc, as one unsigned order.
__device__ __forceinline__ uint64_t cand_key(float s, int32_t pos) {
  return ((uint64_t)score_key(s) << 32) | (uint32_t)(~(uint32_t)pos);
}
__device__ __forceinline__ int32_t cand_pos_of(uint64_t key) {
  return (int32_t)(~(uint32_t)(key & 0xFFFFFFFFull));
}

// ---- Top-K row header (workspace) -----------------------------------------
struct TopkHdr {
  uint32_t cnt;       // candidates appended by the compaction
  uint32_t overflow;  // 1 = more than kCandCap would qualify: use the slow path
  uint32_t done;      // CTAs of this row that have flushed their histogram
  int32_t vbin;       // threshold bin of the level-0 histogram
};
constexpr int kTkThreads = 256;

// Threshold bin of a 4096-bin histogram (counted from the top): the highest
// bin v with (keys in bins >= v) >= k, or bin 0 when the row holds fewer than
// k keys; *out_ge = keys in bins >= v. Every thread of the block must call it
// (it synchronises); the first kTkThreads threads do the work.
__device__ __forceinline__ void find_threshold_bin(const uint32_t* __restrict__ h, int k, int* out_bin,
                                                   uint32_t* out_ge) {
  __shared__ uint32_t warp_tot[kTkThreads / 32];
  __shared__ int s_bin;
  __shared__ uint32_t s_ge;
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const bool act = tid < kTkThreads;
  const int hi = kHistBins - 16 * tid;  // this thread's bins [hi-16, hi), counted from the top
  uint32_t loc = 0;
  if (act) {
#pragma unroll
    for (int i = 1; i <= 16; ++i) loc += h[hi - i];
  }
  uint32_t incl = loc;                   // inclusive scan inside the warp
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const uint32_t v = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += v;
  }
  if (act && lane == 31) warp_tot[wid] = incl;
  if (tid == 0) { s_bin = 0; s_ge = 0xFFFFFFFFu; }
  __syncthreads();
  if (act) {
    uint32_t before = 0, total = 0;
#pragma unroll
    for (int w = 0; w < kTkThreads / 32; ++w) {
      const uint32_t x = warp_tot[w];
      before += w < wid ? x : 0u;
      total += x;
    }
    incl += before;
    const uint32_t excl = incl - loc;
    if (total < (uint32_t)k) {
      if (tid == 0) { s_bin = 0; s_ge = total; }
    } else if (excl < (uint32_t)k && incl >= (uint32_t)k) {
      uint32_t run = excl;
      for (int i = 1; i <= 16; ++i) {
        run += h[hi - i];
        if (run >= (uint32_t)k) { s_bin = hi - i; s_ge = run; break; }
      }
    }
  }
  __syncthreads();
  *out_bin = s_bin;
  *out_ge = s_ge;
}

// End of a histogram-producing CTA: add the CTA's shared histogram into the
// row's global one; the last CTA of the row to finish (counted with an
// atomic, no waiting) derives the threshold bin and the overflow flag for
// the compaction step. `sh` is reused as scratch. Every thread calls it.
__device__ __forceinline__ void topk_hist_flush(uint32_t* sh, uint32_t* __restrict__ ghist, TopkHdr* hdr,
                                                int k, unsigned ctas_in_row) {
  __shared__ int s_last;
  __syncthreads();
  for (int i = threadIdx.x; i < kHistBins; i += blockDim.x) {
    const uint32_t v = sh[i];
    if (v) atomicAdd(ghist + i, v);
  }
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) s_last = (atomicAdd(&hdr->done, 1u) == ctas_in_row - 1);
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  for (int i = threadIdx.x; i < kHistBins; i += blockDim.x) sh[i] = __ldcg(ghist + i);
  __syncthreads();
  int vbin;
  uint32_t ge;
  find_threshold_bin(sh, k, &vbin, &ge);
  if (threadIdx.x == 0) {
    hdr->vbin = vbin;
    hdr->overflow = ge > (uint32_t)kCandCap ? 1u : 0u;
    hdr->cnt = 0;            // a scan may have used it to hand out tiles; the compaction counts from 0
  }
}

// ---- FP8 / FP4 conversions (hardware RNE, satfinite) -----------------------
// Two fp32 -> E4M3 bytes; `lo` lands in the low byte.
__device__ __forceinline__ uint16_t cvt_e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}
__device__ __forceinline__ uint8_t cvt_e4m3(float v) { return (uint8_t)(cvt_e4m3x2(v, 0.f) & 0xFF); }

// Eight non-negative fp32 -> eight E2M1 codes packed low-nibble-first.
__device__ __forceinline__ uint32_t cvt_e2m1x8(const float* f) {
  uint32_t r;
  asm("{\n .reg .b8 b0, b1, b2, b3;\n"
      "cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n"
      "cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n"
      "cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n"
      "cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n"
      "mov.b32 %0, {b0, b1, b2, b3};\n}"
      : "=r"(r)
      : "f"(f[0]), "f"(f[1]), "f"(f[2]), "f"(f[3]), "f"(f[4]), "f"(f[5]), "f"(f[6]), "f"(f[7]));
  return r;
}

// E4M3 byte -> fp32 (exact).
__device__ __forceinline__ float e4m3_to_f32(uint8_t b) {
  uint32_t h2;
  uint16_t v = b;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(v));
  return __half2float(__ushort_as_half((unsigned short)(h2 & 0xFFFF)));
}

// One byte of two E2M1 codes -> f16x2 (low nibble -> low half), exact.
__device__ __forceinline__ uint32_t e2m1x2_to_f16x2(uint32_t byte) {
  uint32_t r;
  uint16_t v = (uint16_t)byte;
  asm("{\n .reg .b8 t, u;\n mov.b16 {t, u}, %1;\n cvt.rn.f16x2.e2m1x2 %0, t;\n}" : "=r"(r) : "h"(v));
  return r;
}

// ---- global loads ----------------------------------------------------------
__device__ __forceinline__ uint4 ldg_stream(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
  return v;
}

// ---- tensor-core MMA (warp-synchronous mma.sync) ----------------------------
// D += A(16x32 e4m3, row) * B(32x8 e4m3, col), fp32 accumulate.
__device__ __forceinline__ void mma_e4m3_16832(float* d, uint32_t a0, uint32_t a1, uint32_t a2,
                                               uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k32.row.col.f32.e4m3.e4m3.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// ---- shared memory helpers -------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

// L2 residency hints: rows that will be read again (the FP4 cache under a
// prefill chunk) are kept, streams read or written once are evicted first.
__device__ __forceinline__ uint64_t l2_evict_first() {
  uint64_t p;
  asm("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint64_t l2_evict_last() {
  uint64_t p;
  asm("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ void st_global_hint(void* p, uint4 v, uint64_t pol) {
  asm volatile("st.global.L1::no_allocate.L2::cache_hint.v4.b32 [%0], {%1,%2,%3,%4}, %5;"
               ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w), "l"(pol) : "memory");
}

}  // namespace csa2
