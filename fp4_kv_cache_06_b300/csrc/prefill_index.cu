// prefill_index.cu — the prefill indexer as a tcgen05 FP8 GEMM.
//
// [CSA2] wire.sakhanda.co, "DeepSeek AI выпустила DeepSeek-V4.1-Flash ...",
//        section "Сжатое разреженное внимание 2 (CSA2)": the encoder's Full
//        layers score the compressed main-KV entries with the indexer and
//        select Top-512 per query; the encoder runs CSA2 at compression
//        ratio 2. Score form taken by this library (the pages give none):
//        s[q][j] = sum_h w[q][h] * relu(qI[q][h] . kI[j]).
//
// For a prefill chunk every query needs the scores of (almost) every entry,
// so the scan becomes a dense GEMM: (entries x 128) . (queries*heads x 128)^T
// in FP8 E4M3 with fp32 accumulation, followed by the relu / head-weight sum.
// Layout (swap-AB): the MMA's M = 128 entries (one TMEM lane each), N = 256 =
// 32 queries x 8 heads (one TMEM column each), K = 128 bytes = 4 MMAs of K 32.
// The head sum is then thread-local in the epilogue and each warp writes 128
// contiguous bytes per query.
//
// CTA = one tile of 32 queries x a contiguous range of 128-entry tiles.
//   warp 0 (one lane): TMA producer, 4-stage ring of 16 KB entry tiles;
//   warp 1: TMEM allocation (512 columns = 2 accumulators of 256) and, on one
//           lane, the MMA issue loop;
//   warps 2..5: epilogue; warp w reads TMEM lanes 32*(w%4).. (its
//           subpartition), so the four warps cover the 128 entries.
// Every wait is bounded; a timeout writes CSA2_ERR_TIMEOUT to d_status and
// the CTA winds down (waiting, again bounded, for its own MMAs) before
// releasing TMEM.
#include <mutex>

#include "common.cuh"
#include "tcgen05.cuh"

namespace csa2 {

constexpr int kPQ = 32;                 // queries per CTA tile
constexpr int kPH = 8;                  // indexer heads (N = kPQ * kPH = 256)
constexpr int kPN = kPQ * kPH;
constexpr int kPM = 128;                // entries per tile (MMA M)
constexpr int kPK = 128;                // indexer dim in bytes (MMA K total)
constexpr int kPStages = 4;
constexpr int kPThreads = 192;          // 6 warps
constexpr uint32_t kPTileBytes = kPM * kPK;       // 16 KB
constexpr uint32_t kPQBytes = kPN * kPK;          // 32 KB

struct PrefillSmem {
  // offsets from a 1024-aligned base
  static constexpr int kQ = 0;                                   // 32 KB
  static constexpr int kA = kQ + kPQBytes;                       // 4 x 16 KB
  static constexpr int kW = kA + kPStages * kPTileBytes;         // 32 x 8 floats
  static constexpr int kBar = kW + kPQ * kPH * 4;                // mbarriers
  static constexpr int kNumBars = 2 * kPStages + 4 + 1;
  static constexpr int kTmemSlot = kBar + kNumBars * 8;
  static constexpr int kFlag = kTmemSlot + 8;
  // + alignment slack; padded past half the SM's shared memory so that one
  // CTA (holding all 512 TMEM columns) runs per SM
  static constexpr int kBytes = (kFlag + 8 + 1024) > 120 * 1024 ? (kFlag + 8 + 1024) : 120 * 1024;
};

__global__ void __launch_bounds__(kPThreads, 1) k_prefill_index(
    const __grid_constant__ CUtensorMap map_k, const __grid_constant__ CUtensorMap map_q,
    const float* __restrict__ w, int Q, int64_t n_keys, int tiles_per_cta, float* __restrict__ scores,
    int64_t stride, int32_t* st, uint64_t wait_ns, int fault) {
  extern __shared__ unsigned char smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023) & ~1023u;
  unsigned char* sp = smem_raw + (base - raw);
  using L = PrefillSmem;
  float* sW = reinterpret_cast<float*>(sp + L::kW);
  volatile int* s_abort = reinterpret_cast<volatile int*>(sp + L::kFlag);
  const uint32_t bar_full = base + L::kBar;                 // [kPStages]
  const uint32_t bar_empty = bar_full + 8 * kPStages;       // [kPStages]
  const uint32_t bar_tfull = bar_empty + 8 * kPStages;      // [2]
  const uint32_t bar_tempty = bar_tfull + 16;               // [2]
  const uint32_t bar_q = bar_tempty + 16;
  const uint32_t tmem_slot = base + L::kTmemSlot;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int qt = blockIdx.y;
  const int64_t n_tiles_total = (n_keys + kPM - 1) / kPM;
  const int64_t t0 = (int64_t)blockIdx.x * tiles_per_cta;
  const int64_t t1 = min(t0 + (int64_t)tiles_per_cta, n_tiles_total);
  const int nt = t1 > t0 ? (int)(t1 - t0) : 0;

  for (int i = tid; i < kPQ * kPH; i += kPThreads) {
    const int q = qt * kPQ + i / kPH;
    sW[i] = q < Q ? w[(int64_t)q * kPH + (i % kPH)] : 0.f;
  }
  if (tid == 0) {
    *s_abort = 0;
    for (int i = 0; i < kPStages; ++i) {
      tc::mbar_init(bar_full + 8 * i, 1);
      tc::mbar_init(bar_empty + 8 * i, 1);
    }
    for (int i = 0; i < 2; ++i) {
      tc::mbar_init(bar_tfull + 8 * i, 1);
      tc::mbar_init(bar_tempty + 8 * i, 128);
    }
    tc::mbar_init(bar_q, 1);
    tc::fence_barrier_init();
  }
  if (warp == 1) {
    tc::tmem_alloc(tmem_slot, 512);
    tc::tmem_relinquish();
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(sp + L::kTmemSlot);

  if (warp == 0 && lane == 0 && nt > 0) {
    // ---- producer
    tc::prefetch_tmap(&map_k);
    tc::prefetch_tmap(&map_q);
    tc::mbar_expect_tx(bar_q, kPQBytes);
    tc::tma_load_2d(base + L::kQ, &map_q, 0, qt * kPN, bar_q);
    for (int i = 0; i < nt; ++i) {
      const int s = i % kPStages;
      if (!tc::mbar_wait(bar_empty + 8 * s, ((i / kPStages) & 1) ^ 1, wait_ns)) {
        report(st, CSA2_ERR_TIMEOUT);
        *s_abort = 1;
        break;
      }
      if (*s_abort) break;
      // fault injection (tests of the bounded waits): the second tile is
      // never loaded nor signalled, so the MMA issuer's wait on it runs out
      if (fault && i == 1) break;
      tc::mbar_expect_tx(bar_full + 8 * s, kPTileBytes);
      tc::tma_load_2d(base + L::kA + s * kPTileBytes, &map_k, 0, (int)((t0 + i) * kPM), bar_full + 8 * s);
    }
  } else if (warp == 1 && lane == 0 && nt > 0) {
    // ---- MMA issuer
    const uint32_t idesc = tc::instr_desc(tc::kFmtE4M3, tc::kFmtE4M3, 0, 0, kPM, kPN);
    bool ok = tc::mbar_wait(bar_q, 0, wait_ns);
    int issued = 0;
    for (int i = 0; ok && i < nt; ++i) {
      const int s = i % kPStages, acc = i & 1;
      if (!tc::mbar_wait(bar_full + 8 * s, (i / kPStages) & 1, wait_ns)) { ok = false; break; }
      if (!tc::mbar_wait(bar_tempty + 8 * acc, ((i >> 1) & 1) ^ 1, wait_ns)) { ok = false; break; }
      if (*s_abort) { ok = false; break; }
      tc::tc_fence_after();
      const uint32_t a0 = base + L::kA + s * kPTileBytes, b0 = base + L::kQ;
#pragma unroll
      for (int kk = 0; kk < kPK / 32; ++kk) {
        const uint64_t ad = tc::smem_desc(a0 + kk * 32, 16, 1024, tc::kSwizzle128B);
        const uint64_t bd = tc::smem_desc(b0 + kk * 32, 16, 1024, tc::kSwizzle128B);
        tc::mma_f8f6f4(tmem + acc * kPN, ad, bd, idesc, kk > 0 ? 1u : 0u);
      }
      tc::mma_commit(bar_empty + 8 * s);
      tc::mma_commit(bar_tfull + 8 * acc);
      issued = i + 1;
    }
    if (!ok) { report(st, CSA2_ERR_TIMEOUT); *s_abort = 1; }
    // wind down: the last commit of each accumulator tells that its MMAs finished
    if (issued > 0) {
      const int last = issued - 1;
      tc::mbar_wait(bar_tfull + 8 * (last & 1), (last >> 1) & 1, wait_ns);
    }
  } else if (warp >= 2) {
    // ---- epilogue: lane = entry, columns = query*8 + head
    const int sub = warp & 3;
    for (int i = 0; i < nt; ++i) {
      const int acc = i & 1;
      // warp-uniform decision: the TMEM loads below are warp-collective
      const bool got = tc::mbar_wait(bar_tfull + 8 * acc, (i >> 1) & 1, wait_ns);
      if (!__all_sync(0xffffffffu, got) || __any_sync(0xffffffffu, *s_abort != 0)) {
        if (lane == 0) { report(st, CSA2_ERR_TIMEOUT); *s_abort = 1; }
        break;
      }
      tc::tc_fence_after();
      const int64_t key = (t0 + i) * kPM + sub * 32 + lane;
      const uint32_t taddr = tmem + ((uint32_t)(sub * 32) << 16) + acc * kPN;
      float out[kPQ];
#pragma unroll
      for (int c = 0; c < kPN / 32; ++c) {
        uint32_t r[32];
        tc::tmem_ld32(taddr + c * 32, r);
        tc::tmem_ld_wait();
#pragma unroll
        for (int qq = 0; qq < 4; ++qq) {
          float sacc = 0.f;
#pragma unroll
          for (int h = 0; h < kPH; ++h)
            sacc = fmaf(sW[(c * 4 + qq) * kPH + h], fmaxf(__uint_as_float(r[qq * kPH + h]), 0.f), sacc);
          out[c * 4 + qq] = sacc;
        }
      }
      tc::tc_fence_before();
      tc::mbar_arrive(bar_tempty + 8 * acc);
      if (key < n_keys) {
#pragma unroll
        for (int qq = 0; qq < kPQ; ++qq) {
          const int q = qt * kPQ + qq;
          if (q < Q) scores[(int64_t)q * stride + key] = out[qq];
        }
      }
    }
  }
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem, 512);
  }
}

// ---- host -----------------------------------------------------------------------
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
  static std::mutex mu;
  static EncodeTiledFn fn = nullptr;
  std::lock_guard<std::mutex> lk(mu);
  if (fn == nullptr) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

bool make_tmap_rows128(CUtensorMap* map, const void* base, uint64_t rows, uint64_t row_bytes, uint32_t box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr || rows == 0 || (row_bytes & 15) || (reinterpret_cast<uintptr_t>(base) & 15)) return false;
  cuuint64_t dims[2] = {row_bytes, rows};
  cuuint64_t strides[1] = {row_bytes};
  cuuint32_t box[2] = {128, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int prefill_init_attributes() {
  if (cudaFuncSetAttribute(k_prefill_index, cudaFuncAttributeMaxDynamicSharedMemorySize, PrefillSmem::kBytes) !=
      cudaSuccess)
    return CSA2_ERR_CUDA;
  return CSA2_OK;
}

int launch_prefill_index(const uint8_t* qI, const float* w, int Q, const uint8_t* kI, int64_t n_keys, float* scores,
                         int64_t stride, int32_t* st, cudaStream_t s) {
  if (Q == 0 || n_keys == 0) return CSA2_OK;
  CUtensorMap mk, mq;
  if (!make_tmap_rows128(&mk, kI, (uint64_t)n_keys, kPK, kPM)) return CSA2_ERR_INVALID_ARG;
  if (!make_tmap_rows128(&mq, qI, (uint64_t)Q * kPH, kPK, kPN)) return CSA2_ERR_INVALID_ARG;
  const int qtiles = (Q + kPQ - 1) / kPQ;
  const int64_t ktiles = (n_keys + kPM - 1) / kPM;
  // split the entry tiles so the grid covers the 148 SMs a few times
  int64_t splits = (4 * kSMs + qtiles - 1) / qtiles;
  if (splits > ktiles) splits = ktiles;
  if (splits < 1) splits = 1;
  const int tpc = (int)((ktiles + splits - 1) / splits);
  splits = (ktiles + tpc - 1) / tpc;
  dim3 grid((unsigned)splits, (unsigned)qtiles);
  k_prefill_index<<<grid, kPThreads, PrefillSmem::kBytes, s>>>(mk, mq, w, Q, n_keys, tpc, scores, stride, st,
                                                                debug_wait_ns(), debug_fault() == kFaultPrefill);
  count_launch();
  return launch_status();
}

}  // namespace csa2
