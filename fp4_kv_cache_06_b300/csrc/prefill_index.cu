// prefill_index.cu — the prefill indexer: a tcgen05 FP8 GEMM with the Top-K
// candidate selection fused into its epilogue.
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
// The head sum is then thread-local in the epilogue.
//
// One persistent kernel, one CTA per SM. The work is the list of units
// (query tile of 32, entry tile of 128) that some query of the tile can see
// (causally invisible tiles are not in the list); each CTA takes one
// contiguous, equal share of it, so a CTA meets at most a few query tiles in
// a row ("segments"), each loaded once into one of two query buffers.
//   warp 0 (one lane): TMA producer (query tiles: 2 buffers; entry tiles:
//           4-stage ring of 16 KB);
//   warp 1: TMEM allocation (512 columns = 2 accumulators of 256) and, on one
//           lane, the MMA issue loop;
//   warps 2..17: epilogue. TMEM lane subpartition warp % 4, column quarter
//           (warp - 2) / 4: 32 entries x 8 queries per warp and tile, read
//           in 16-column chunks (the next chunk loads while one is summed);
//           relu and the head weights as paired fp32x2 FMAs.
// Modes:
//   write  — the score of every entry of a unit at scores[q][col];
//   filter — an entry whose score is at or above its query's threshold
//            becomes a candidate: its unique 64-bit key (score key,
//            ~position) goes to the query's list. A warp fills each of its
//            queries' lists in chunks of 32 slots, with the next chunk
//            reserved ahead, so no append waits on an atomic; slots left
//            unfilled are holes (key 0), counted in the list header.
//
// Selection for a prefill chunk (launch_prefill_candidates, then
// launch_prefill_finish):
//   1. sampled pass (write mode): the scores of every S-th entry tile
//      (S >= 16, at most 16 sampled tiles: 2048 entries);
//   2. threshold: per query, the score key of the r-th best visible sampled
//      score, r chosen so that about 2048 visible entries are expected at or
//      above it (a warp bisection over register-held keys). A query with at
//      most kCandCap visible entries takes all of them (threshold key 0);
//   3. filter pass over every visible unit;
//   4. check: a query with fewer candidates than min(k, visible), or more
//      than its list holds, is marked (the Top-K's overflow flag), and so is
//      its query tile; the marked tiles' rows are then written in full
//      (write mode over those tiles only);
//   5. exact selection: over each unmarked query's list (a warp; bisection on
//      register-held score keys, the radix select when a tie at the boundary
//      score must be split by position), and over each marked query's full
//      row (a warp; radix select).
// In the common case nothing but ~2048 candidates per query is written.
//
// Every wait is bounded; a timeout writes CSA2_ERR_TIMEOUT to d_status and
// the CTA winds down (waiting, again bounded, for its own MMAs) before
// releasing TMEM.
#include <mutex>

#include "common.cuh"
#include "tcgen05.cuh"

namespace csa2 {

constexpr int kPQ = 32;                 // queries per query tile
constexpr int kPH = 8;                  // indexer heads (N = kPQ * kPH = 256)
constexpr int kPN = kPQ * kPH;
constexpr int kPM = 128;                // entries per tile (MMA M)
constexpr int kPK = 128;                // indexer dim in bytes (MMA K total)
constexpr int kPStages = 4;
constexpr int kPEpiWarps = 16;
constexpr int kPThreads = 64 + 32 * kPEpiWarps;   // producer, MMA, 16 epilogue warps
constexpr int kPQw = kPQ * 4 / kPEpiWarps;        // queries per epilogue warp (8)
constexpr uint32_t kPTileBytes = kPM * kPK;       // 16 KB
constexpr uint32_t kPQBytes = kPN * kPK;          // 32 KB
constexpr int kPMaxQTiles = 2048;                 // query tiles per launch (the unit table)
constexpr int kPSampleMin = 16;                   // sampled pass: every S-th entry tile, S >= 16,
constexpr int kPSampleTiles = 16;                 //   at most 16 sampled tiles (2048 entries)
constexpr int kPCandTarget = 2048;                // candidates expected per query
constexpr int kPChunk = 32;                       // candidate-list slots reserved per warp and query at a time
constexpr int kPSelWarps = 4;                     // selection kernels: one warp per query (32 KB)
constexpr int kPSelBins = 2048;                   // radix digits of 11 bits (a warp's histogram)

enum PrefillMode : int { kPWrite = 0, kPFilter = 1 };

// The Top-K library's workspace (topk.cu): row headers and candidate lists.
int topk_prepare(void* ws, int B, cudaStream_t s);
TopkHdr* topk_ws_hdr(void* ws, int B);
uint64_t* topk_ws_cand(void* ws, int B);
static size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

struct PrefillPass {
  const float* w;
  const int64_t* n_vis;     // nullable: every entry is visible to every query
  const int32_t* gate;      // nullable: query tiles whose gate is 0 have no units
  float* scores;            // write mode: scores[q * stride + col]
  int64_t stride;
  const uint32_t* tau;      // filter mode: per-query threshold key
  TopkHdr* hdr;             //   candidate counts
  uint64_t* cand;           //   candidate lists [Q][kCandCap]
  int32_t* st;
  uint64_t wait_ns;
  int64_t n_keys;
  int64_t seq_tiles;        // tiles in this pass's sequence; tile t covers entries from t * tile_step * 128
  int Q, qt0, qtiles;       // query tiles qt0 .. qt0 + qtiles - 1
  int tile_step;
  int mode, fault;
};

struct PrefillSmem {
  // offsets from a 1024-aligned base
  static constexpr int kQ = 0;                                   // 2 x 32 KB query tiles
  static constexpr int kA = kQ + 2 * kPQBytes;                   // 4 x 16 KB entry tiles
  static constexpr int kW = kA + kPStages * kPTileBytes;         // per epilogue warp: its queries' head weights
  static constexpr int kTau = kW + kPEpiWarps * kPQw * kPH * 4;   // per epilogue warp: threshold scores
  static constexpr int kVis = kTau + kPEpiWarps * kPQw * 4;        //   and visible counts of its queries
  static constexpr int kPre = kVis + kPEpiWarps * kPQw * 4;        // unit table: int64 [kPMaxQTiles + 1]
  static constexpr int kBar = kPre + (kPMaxQTiles + 1) * 8;
  static constexpr int kNumBars = 2 * kPStages + 2 + 2 + 2 + 2;  // full/empty, tfull/tempty, qfull/qempty
  static constexpr int kTmemSlot = kBar + kNumBars * 8;
  static constexpr int kFlag = kTmemSlot + 8;
  static constexpr int kBytes = kFlag + 8 + 1024;                // + alignment slack (> half the SM: 1 CTA)
};
static_assert(PrefillSmem::kBar % 8 == 0, "mbarriers need 8-byte alignment");
static_assert(PrefillSmem::kBytes > 116 * 1024 && PrefillSmem::kBytes <= 227 * 1024,
              "one CTA per SM (it holds all 512 TMEM columns)");

// Walk over a CTA's units: local query tile qi, sequence tile t. pre[i] is the
// number of units of local query tiles before i.
struct UnitWalk {
  const int64_t* pre;
  int qtiles;
  int qi;
  int t, vt;                 // sequence tile within query tile qi, and qi's unit count (< 2^24)
  __device__ void start(int64_t u) {
    int lo = 0, hi = qtiles - 1;                 // last qi with pre[qi] <= u
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (pre[mid] <= u) lo = mid; else hi = mid - 1;
    }
    qi = lo;
    t = (int)(u - pre[qi]);
    vt = (int)(pre[qi + 1] - pre[qi]);
  }
  __device__ bool last_of_tile() const { return t + 1 >= vt; }
  __device__ void next() {
    if (t + 1 >= vt) {
      do { ++qi; } while (qi < qtiles && pre[qi + 1] == pre[qi]);
      t = 0;
      if (qi < qtiles) vt = (int)(pre[qi + 1] - pre[qi]);
    } else {
      ++t;
    }
  }
};

// acc += (w.lo, w.hi) * (relu(d0), relu(d1)) as one fp32x2 FMA. The two
// relu results are formed inside the asm so that they land in a register
// pair; each lane's sum is the same fma as the scalar form.
__device__ __forceinline__ uint64_t relu_fma2(uint64_t acc, uint64_t w2, uint32_t d0, uint32_t d1) {
  asm("{\n .reg .f32 a, b;\n .reg .b64 p;\n"
      " max.f32 a, %2, 0f00000000;\n max.f32 b, %3, 0f00000000;\n"
      " mov.b64 p, {a, b};\n fma.rn.f32x2 %0, %1, p, %0;\n}"
      : "+l"(acc) : "l"(w2), "f"(__uint_as_float(d0)), "f"(__uint_as_float(d1)));
  return acc;
}
__device__ __forceinline__ float sum_f32x2(uint64_t a) {
  float lo, hi;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(a));
  return lo + hi;
}
// 32 lanes x 16 consecutive 32-bit TMEM columns (thread t: lane base + t).
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t* r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}
// tcgen05.wait::ld with the 16 destination registers of the load it waits
// for tied in, so that no use of them can be scheduled before the wait.
__device__ __forceinline__ void tmem_wait_tied16(uint32_t* r) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
                 "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]),
                 "+r"(r[15])
               :
               : "memory");
}
// Threshold key -> the smallest score that has a key at or above it (key 0:
// every score). Scores are finite, so comparing scores with it keeps every
// entry whose key is at or above the threshold (and, at a threshold of +0,
// also -0: an extra candidate, harmless).
__device__ __forceinline__ float key_score(uint32_t key) {
  if (key == 0u) return -INFINITY;
  return __uint_as_float((key & 0x80000000u) ? (key & 0x7FFFFFFFu) : ~key);
}

template <int kMode>
__global__ void __launch_bounds__(kPThreads, 1) k_prefill_index(const __grid_constant__ CUtensorMap map_k,
                                                                 const __grid_constant__ CUtensorMap map_q,
                                                                 const __grid_constant__ PrefillPass a) {
  extern __shared__ unsigned char smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023) & ~1023u;
  unsigned char* sp = smem_raw + (base - raw);
  using L = PrefillSmem;
  int64_t* sPre = reinterpret_cast<int64_t*>(sp + L::kPre);
  volatile int* s_abort = reinterpret_cast<volatile int*>(sp + L::kFlag);
  const uint32_t bar_full = base + L::kBar;                 // [kPStages]
  const uint32_t bar_empty = bar_full + 8 * kPStages;       // [kPStages]
  const uint32_t bar_tfull = bar_empty + 8 * kPStages;      // [2]
  const uint32_t bar_tempty = bar_tfull + 16;               // [2]
  const uint32_t bar_qfull = bar_tempty + 16;               // [2]
  const uint32_t bar_qempty = bar_qfull + 16;               // [2]
  const uint32_t tmem_slot = base + L::kTmemSlot;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t span = (int64_t)a.tile_step * kPM;          // entries between consecutive sequence tiles

  // ---- the unit table: units of local query tile i = its sequence tiles
  //      that start below the largest visible count of its queries
  for (int i = warp; i < a.qtiles; i += kPThreads / 32) {
    const int64_t q = (int64_t)(a.qt0 + i) * kPQ + lane;
    int64_t v = 0;
    if (q < a.Q) {
      v = a.n_vis ? a.n_vis[q] : a.n_keys;
      v = v < 0 ? 0 : (v > a.n_keys ? a.n_keys : v);
    }
    for (int off = 16; off > 0; off >>= 1) {
      const int64_t o = __shfl_xor_sync(0xffffffffu, v, off);
      v = o > v ? o : v;
    }
    int64_t vt = (v + span - 1) / span;
    if (vt > a.seq_tiles) vt = a.seq_tiles;
    if (a.gate && a.gate[a.qt0 + i] == 0) vt = 0;
    if (lane == 0) sPre[i + 1] = vt;
  }
  __syncthreads();
  if (warp == 0) {
    // in-place inclusive prefix over slots 1..qtiles (slot i + 1 holds the
    // count of tile i), so that pre[i] = units before tile i; lane l owns the
    // contiguous slots of tiles [i0, i1) and touches no other
    const int per = (a.qtiles + 31) / 32;
    const int i0 = min(lane * per, a.qtiles), i1 = min(i0 + per, a.qtiles);
    int64_t sum = 0;
    for (int i = i0; i < i1; ++i) sum += sPre[i + 1];
    int64_t incl = sum;
    for (int off = 1; off < 32; off <<= 1) {
      const int64_t o = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += o;
    }
    int64_t run = incl - sum;
    for (int i = i0; i < i1; ++i) {
      run += sPre[i + 1];
      sPre[i + 1] = run;
    }
    if (lane == 0) sPre[0] = 0;
  }
  __syncthreads();
  const int64_t total = sPre[a.qtiles];
  const int64_t share = (total + gridDim.x - 1) / gridDim.x;
  const int64_t u0 = (int64_t)blockIdx.x * share;
  const int64_t u1 = min(u0 + share, total);
  if (u0 >= u1) return;                          // CTA-uniform: nothing allocated yet
  const int nu = (int)(u1 - u0);

  if (tid == 0) {
    *s_abort = 0;
    for (int i = 0; i < kPStages; ++i) {
      tc::mbar_init(bar_full + 8 * i, 1);
      tc::mbar_init(bar_empty + 8 * i, 1);
    }
    for (int i = 0; i < 2; ++i) {
      tc::mbar_init(bar_tfull + 8 * i, 1);
      tc::mbar_init(bar_tempty + 8 * i, 32 * kPEpiWarps);
      tc::mbar_init(bar_qfull + 8 * i, 1);
      tc::mbar_init(bar_qempty + 8 * i, 1);
    }
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
  UnitWalk it{sPre, a.qtiles, 0, 0, 0};
  it.start(u0);

  if (warp == 0 && lane == 0) {
    // ---- producer
    tc::prefetch_tmap(&map_k);
    tc::prefetch_tmap(&map_q);
    int seg = -1, qi_prev = -1;
    for (int i = 0; i < nu; ++i, it.next()) {
      if (it.qi != qi_prev) {                    // a new query tile: into the other query buffer
        ++seg;
        const int qs = seg & 1;
        if (seg >= 2 && !tc::mbar_wait(bar_qempty + 8 * qs, ((seg >> 1) - 1) & 1, a.wait_ns)) {
          report(a.st, CSA2_ERR_TIMEOUT);
          *s_abort = 1;
          break;
        }
        tc::mbar_expect_tx(bar_qfull + 8 * qs, kPQBytes);
        tc::tma_load_2d(base + L::kQ + qs * kPQBytes, &map_q, 0, (a.qt0 + it.qi) * kPN, bar_qfull + 8 * qs);
        qi_prev = it.qi;
      }
      const int s = i % kPStages;
      if (!tc::mbar_wait(bar_empty + 8 * s, ((i / kPStages) & 1) ^ 1, a.wait_ns)) {
        report(a.st, CSA2_ERR_TIMEOUT);
        *s_abort = 1;
        break;
      }
      if (*s_abort) break;
      // fault injection (tests of the bounded waits): the second tile is
      // never loaded nor signalled, so the MMA issuer's wait on it runs out
      if (a.fault && i == 1) break;
      tc::mbar_expect_tx(bar_full + 8 * s, kPTileBytes);
      tc::tma_load_2d(base + L::kA + s * kPTileBytes, &map_k, 0, it.t * (int)span, bar_full + 8 * s);
    }
  } else if (warp == 1 && lane == 0) {
    // ---- MMA issuer
    const uint32_t idesc = tc::instr_desc(tc::kFmtE4M3, tc::kFmtE4M3, 0, 0, kPM, kPN);
    bool ok = true;
    int issued = 0, seg = -1, qi_prev = -1;
    for (int i = 0; i < nu; ++i, it.next()) {
      if (it.qi != qi_prev) {
        ++seg;
        qi_prev = it.qi;
        if (!tc::mbar_wait(bar_qfull + 8 * (seg & 1), (seg >> 1) & 1, a.wait_ns)) { ok = false; break; }
      }
      const int s = i % kPStages, acc = i & 1;
      if (!tc::mbar_wait(bar_full + 8 * s, (i / kPStages) & 1, a.wait_ns)) { ok = false; break; }
      if (!tc::mbar_wait(bar_tempty + 8 * acc, ((i >> 1) & 1) ^ 1, a.wait_ns)) { ok = false; break; }
      if (*s_abort) { ok = false; break; }
      tc::tc_fence_after();
      const uint32_t a0 = base + L::kA + s * kPTileBytes, b0 = base + L::kQ + (seg & 1) * kPQBytes;
#pragma unroll
      for (int kk = 0; kk < kPK / 32; ++kk) {
        const uint64_t ad = tc::smem_desc(a0 + kk * 32, 16, 1024, tc::kSwizzle128B);
        const uint64_t bd = tc::smem_desc(b0 + kk * 32, 16, 1024, tc::kSwizzle128B);
        tc::mma_f8f6f4(tmem + acc * kPN, ad, bd, idesc, kk > 0 ? 1u : 0u);
      }
      tc::mma_commit(bar_empty + 8 * s);
      tc::mma_commit(bar_tfull + 8 * acc);
      if (it.last_of_tile()) tc::mma_commit(bar_qempty + 8 * (seg & 1));   // the query buffer is free
      issued = i + 1;
    }
    if (!ok) { report(a.st, CSA2_ERR_TIMEOUT); *s_abort = 1; }
    // wind down: the last commit of each accumulator tells that its MMAs finished
    if (issued > 0) {
      const int last = issued - 1;
      tc::mbar_wait(bar_tfull + 8 * (last & 1), (last >> 1) & 1, a.wait_ns);
    }
  } else if (warp >= 2) {
    // ---- epilogue: lane = entry, columns = query * 8 + head
    const int e = warp - 2, sub = warp & 3, grp = e >> 2;
    float* sWe = reinterpret_cast<float*>(sp + L::kW) + e * kPQw * kPH;
    float* sTau = reinterpret_cast<float*>(sp + L::kTau) + e * kPQw;      // filter: threshold scores
    int32_t* sVis = reinterpret_cast<int32_t*>(sp + L::kVis) + e * kPQw;  // filter: visible entries
    // Filter: each query's candidates go to its list in chunks of kPChunk
    // slots. cur[qq] is the next free slot of the current chunk (chunk bases
    // are multiples of kPChunk, and a chunk is left as soon as it is full, so
    // cur % kPChunk == 0 means a fresh chunk); pre[qq] (valid in lane 0) is
    // the base of the chunk reserved next, whose atomic is read only at the
    // next change of chunk. Slots reserved but not filled are holes: key 0,
    // counted in the header's `done` word.
    uint32_t cur[kPQw], pre[kPQw];
#pragma unroll
    for (int qq = 0; qq < kPQw; ++qq) { cur[qq] = 0; pre[qq] = 0; }
    int32_t minvis = 0;                         // filter: fewest visible entries of the warp's queries
    float* rowp = a.scores;                     // write: row of the warp's first query
    uint32_t rows_ok = 0;                       // write: bit qq set when query q0 + qq exists
    const int32_t span32 = (int32_t)span, nk32 = (int32_t)a.n_keys;   // both < 2^31
    int qi_prev = -1, q0_prev = 0;
    bool aborted = false;
    // filter: mark the holes of the warp's queries q0 .. (at the end of their tile)
    auto close_lists = [&](int q0) {
#pragma unroll
      for (int qq = 0; qq < kPQw; ++qq) {
        const int q = q0 + qq;
        if (q >= a.Q) break;
        const uint32_t p = __shfl_sync(0xffffffffu, pre[qq], 0);
        const uint32_t room = kPChunk - (cur[qq] & (kPChunk - 1));
        uint64_t* lst = a.cand + (int64_t)q * kCandCap;
        if ((uint32_t)lane < room && cur[qq] + lane < (uint32_t)kCandCap) lst[cur[qq] + lane] = 0ull;
        if (p + lane < (uint32_t)kCandCap) lst[p + lane] = 0ull;
        if (lane == 0) atomicAdd(&a.hdr[q].done, room + kPChunk);
      }
    };
    for (int i = 0; i < nu; ++i, it.next()) {
      const int q0 = (a.qt0 + it.qi) * kPQ + grp * kPQw;      // this warp's first query
      if (it.qi != qi_prev) {
        if (kMode == kPFilter && qi_prev >= 0) close_lists(q0_prev);
        __syncwarp();
        for (int j = lane; j < kPQw * kPH; j += 32) {
          const int q = q0 + j / kPH;
          sWe[j] = q < a.Q ? a.w[(int64_t)q * kPH + (j % kPH)] : 0.f;
        }
        if (kMode == kPFilter) {
          int64_t v = 0;
          float tf = INFINITY;
          uint32_t base = 0;
          if (lane < kPQw && q0 + lane < a.Q) {
            const int q = q0 + lane;
            v = a.n_vis ? a.n_vis[q] : a.n_keys;
            v = v < 0 ? 0 : (v > a.n_keys ? a.n_keys : v);
            tf = key_score(a.tau[q]);
            base = atomicAdd(&a.hdr[q].cnt, 2u * kPChunk);       // the first chunk and the next
          }
          if (lane < kPQw) { sVis[lane] = (int32_t)v; sTau[lane] = tf; }
          int64_t mv = lane < kPQw ? v : a.n_keys;
          for (int off = 16; off > 0; off >>= 1) {
            const int64_t o = __shfl_xor_sync(0xffffffffu, mv, off);
            mv = o < mv ? o : mv;
          }
          minvis = (int32_t)mv;
#pragma unroll
          for (int qq = 0; qq < kPQw; ++qq) {
            cur[qq] = __shfl_sync(0xffffffffu, base, qq);
            pre[qq] = cur[qq] + kPChunk;
          }
        }
        if (kMode == kPWrite) {
          rowp = a.scores + (int64_t)q0 * a.stride;
          rows_ok = 0;
#pragma unroll
          for (int qq = 0; qq < kPQw; ++qq) rows_ok |= (q0 + qq < a.Q ? 1u : 0u) << qq;
        }
        __syncwarp();
        qi_prev = it.qi;
        q0_prev = q0;
      }
      const int acc = i & 1;
      // warp-uniform decision: the TMEM loads below are warp-collective. A
      // role that stopped (timeout) stops the commits, so this wait then runs
      // out as well; no separate abort check is needed on the way.
      const uint32_t tf_bar = bar_tfull + 8 * acc, tf_par = (i >> 1) & 1;
      const bool got = tc::mbar_try_wait(tf_bar, tf_par) || tc::mbar_wait(tf_bar, tf_par, a.wait_ns);
      if (!__all_sync(0xffffffffu, got)) {
        if (lane == 0) { report(a.st, CSA2_ERR_TIMEOUT); *s_abort = 1; }
        aborted = true;
        break;
      }
      tc::tc_fence_after();
      const int32_t tb = it.t * span32;                                  // the tile's first entry
      const int32_t entry = tb + sub * 32 + lane;                        // < n_keys + 128 <= 2^31 - 1
      const int32_t col = it.t * kPM + sub * 32 + lane;
      const bool fullvis = tb + kPM <= minvis;                           // filter: no entry past any limit
      const uint32_t taddr = tmem + ((uint32_t)(sub * 32) << 16) + acc * kPN + grp * (kPQw * kPH);
      // four 16-column chunks (2 queries each): chunk c + 1 is read from TMEM
      // while chunk c is summed; the accumulator is handed back once the last
      // chunk has arrived in registers
      uint32_t ra[16], rb[16];
      float scv[kPQw];
      tmem_ld16(taddr, ra);
      tmem_wait_tied16(ra);
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t* cu = (c & 1) ? rb : ra;
        uint32_t* nx = (c & 1) ? ra : rb;
        if (c < 3) tmem_ld16(taddr + (c + 1) * 16, nx);
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const ulonglong2* wv = reinterpret_cast<const ulonglong2*>(sWe + (c * 2 + j) * kPH);
          const ulonglong2 wa = wv[0], wb = wv[1];
          const uint32_t* d = cu + j * kPH;
          uint64_t acc2 = 0ull;
          acc2 = relu_fma2(acc2, wa.x, d[0], d[1]);
          acc2 = relu_fma2(acc2, wa.y, d[2], d[3]);
          acc2 = relu_fma2(acc2, wb.x, d[4], d[5]);
          acc2 = relu_fma2(acc2, wb.y, d[6], d[7]);
          scv[c * 2 + j] = sum_f32x2(acc2);
        }
        if (c < 3) tmem_wait_tied16(nx);
        if (c == 2) {                                       // all of the tile is in registers
          tc::tc_fence_before();
          tc::mbar_arrive(bar_tempty + 8 * acc);
        }
      }
      {
        if (kMode == kPWrite) {
          float* pc = rowp + col;
          const bool inside = tb + kPM <= nk32 || entry < nk32;
#pragma unroll
          for (int qq8 = 0; qq8 < 8; ++qq8)
            if (((rows_ok >> qq8) & 1u) && inside) pc[(int64_t)qq8 * a.stride] = scv[qq8];
        } else {
          const float4 ta = reinterpret_cast<const float4*>(sTau)[0];
          const float4 tb = reinterpret_cast<const float4*>(sTau)[1];
          uint32_t take = (scv[0] >= ta.x ? 1u : 0u) | (scv[1] >= ta.y ? 2u : 0u) | (scv[2] >= ta.z ? 4u : 0u) |
                          (scv[3] >= ta.w ? 8u : 0u) | (scv[4] >= tb.x ? 16u : 0u) | (scv[5] >= tb.y ? 32u : 0u) |
                          (scv[6] >= tb.z ? 64u : 0u) | (scv[7] >= tb.w ? 128u : 0u);
          if (!fullvis) {
#pragma unroll
            for (int qq8 = 0; qq8 < 8; ++qq8)
              if (entry >= sVis[qq8]) take &= ~(1u << qq8);
          }
          if (__any_sync(0xffffffffu, take != 0)) {
#pragma unroll
            for (int qq8 = 0; qq8 < 8; ++qq8) {
              const int qq = qq8;
              const bool t = (take >> qq8) & 1u;
              const uint32_t bal = __ballot_sync(0xffffffffu, t);
              if (bal == 0u) continue;
              const uint32_t n = __popc(bal), rk = __popc(bal & ((1u << lane) - 1u));
              const uint32_t room = kPChunk - (cur[qq] & (kPChunk - 1));
              uint32_t p = 0;
              if (n >= room) p = __shfl_sync(0xffffffffu, pre[qq], 0);     // this batch reaches the next chunk
              if (t) {
                const uint32_t slot = rk < room ? cur[qq] + rk : p + (rk - room);
                if (slot < (uint32_t)kCandCap) a.cand[(int64_t)(q0 + qq) * kCandCap + slot] = cand_key(scv[qq8], entry);
              }
              if (n < room) {
                cur[qq] += n;
              } else {
                cur[qq] = p + (n - room);
                uint32_t nb = 0;
                if (lane == 0) nb = atomicAdd(&a.hdr[q0 + qq].cnt, (uint32_t)kPChunk);   // read at the next change
                pre[qq] = nb;
              }
            }
          }
        }
      }
    }
    if (kMode == kPFilter && !aborted && qi_prev >= 0) close_lists(q0_prev);
  }
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem, 512);
  }
}

// ---- per-query selection: one warp, exact radix select ------------------------
// Key sources: key = (score key << 32) | ~position, unique per entry, so the
// best entries by (score descending, position ascending) are the largest keys.
struct RowSource {               // a full score row: entry i has score s[i]
  const float* s;
  int n;
  __device__ bool get(int i, uint64_t& key) const { key = cand_key(s[i], i); return true; }
};
struct SampleSource {            // sampled column i holds entry (i / 128) * step * 128 + i % 128
  const float* s;
  int n;
  int64_t step, vis;
  __device__ bool get(int i, uint64_t& key) const {
    const int64_t entry = (int64_t)(i / kPM) * step * kPM + (i % kPM);
    if (entry >= vis) return false;
    key = cand_key(s[i], (int32_t)entry);
    return true;
  }
};

// Warp-wide: a key thr such that exactly kth keys of the source are >= thr
// (1 <= kth <= number of keys; keys are distinct), by MSD radix passes of up
// to 11 bits. The bits every key shares are skipped first, and the passes
// stop as soon as the keys at or above the digit found number exactly kth
// (thr then has zeros below that digit). With hi_only they stop at the
// score word: thr's high word is then the score key of the kth largest, and
// at least kth keys have a score key >= it. h: kPSelBins words of shared
// memory owned by the warp.
// Calls fn(key) for every key of the source that lane `lane` owns (entries
// lane, lane + 32, ...), eight loads in flight at a time.
template <class Src, class Fn>
__device__ __forceinline__ void for_keys(const Src& src, int lane, Fn fn) {
  for (int i0 = 0; i0 < src.n; i0 += 32 * 8) {
    uint64_t kk[8];
    bool ok[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int i = i0 + u * 32 + lane;
      ok[u] = i < src.n && src.get(i, kk[u]);
    }
#pragma unroll
    for (int u = 0; u < 8; ++u)
      if (ok[u]) fn(kk[u]);
  }
}

template <class Src>
__device__ uint64_t warp_kth(const Src& src, int kth, bool hi_only, uint32_t* h, int lane) {
  unsigned long long all_and = ~0ull, all_or = 0ull;
  for_keys(src, lane, [&](uint64_t key) { all_and &= key; all_or |= key; });
  for (int off = 16; off > 0; off >>= 1) {
    all_and &= __shfl_xor_sync(0xffffffffu, all_and, off);
    all_or |= __shfl_xor_sync(0xffffffffu, all_or, off);
  }
  const uint64_t diff = all_and ^ all_or;
  if (diff == 0ull) return all_and;                 // a single key
  int hi_bit = 63 - __clzll((long long)diff);       // the highest bit that differs
  uint64_t mask = hi_bit < 63 ? ~((2ull << hi_bit) - 1) : 0ull;
  uint64_t prefix = all_and & mask;
  int rem = kth;
  while (hi_bit >= (hi_only ? 32 : 0)) {
    const int width = hi_bit + 1 < 11 ? hi_bit + 1 : 11;
    const int shift = hi_bit + 1 - width;
    const uint32_t nb = 1u << width;
    for (uint32_t b = lane; b < (uint32_t)kPSelBins; b += 32) h[b] = 0;
    __syncwarp();
    for_keys(src, lane, [&](uint64_t key) {
      if ((key & mask) == prefix) atomicAdd(&h[(uint32_t)(key >> shift) & (nb - 1)], 1u);
    });
    __syncwarp();
    // lane l owns the digits [kPSelBins - 64 (l + 1), kPSelBins - 64 l) of
    // a 2048-digit range, counted from the top (digits >= nb are empty)
    constexpr int per = kPSelBins / 32;
    uint32_t loc = 0;
    for (int j = 0; j < per; ++j) loc += h[kPSelBins - 1 - per * lane - j];
    uint32_t incl = loc;
    for (int off = 1; off < 32; off <<= 1) {
      const uint32_t o = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += o;
    }
    const uint32_t excl = incl - loc;
    uint32_t dgt = 0, at_dgt = 0, above = 0;
    const bool mine = excl < (uint32_t)rem && incl >= (uint32_t)rem;
    if (mine) {
      uint32_t run = excl;
      for (int j = 0; j < per; ++j) {
        const uint32_t d = kPSelBins - 1 - per * lane - j;
        const uint32_t c = h[d];
        if (run + c >= (uint32_t)rem) { dgt = d; at_dgt = c; above = run; break; }
        run += c;
      }
    }
    const int owner = __ffs(__ballot_sync(0xffffffffu, mine)) - 1;
    dgt = __shfl_sync(0xffffffffu, dgt, owner);
    at_dgt = __shfl_sync(0xffffffffu, at_dgt, owner);
    above = __shfl_sync(0xffffffffu, above, owner);
    __syncwarp();
    rem -= (int)above;
    prefix |= (uint64_t)dgt << shift;
    mask |= (uint64_t)(nb - 1) << shift;
    if (at_dgt == (uint32_t)rem) break;             // every key of this digit is among the kth best
    hi_bit = shift - 1;
  }
  return prefix;
}

// Warp-wide: the kth largest of the lanes' register-held score keys (key 0 =
// absent; a score's key is never 0), by bisection on the key bits: the
// largest K with at least kth keys >= K. Keys u >= nu (a warp-uniform bound,
// in groups of 16) are all absent and skipped; so are the bits above the
// highest bit in which the present keys differ. No shared memory, no atomics.
template <int N>
__device__ __forceinline__ uint32_t warp_count_ge(const uint32_t (&key)[N], uint32_t c, int nu) {
  uint32_t cnt = 0;
#pragma unroll
  for (int g = 0; g < N; g += 16) {
    if (g < nu) {
#pragma unroll
      for (int u = g; u < g + 16 && u < N; ++u) cnt += key[u] >= c ? 1u : 0u;
    }
  }
  return __reduce_add_sync(0xffffffffu, cnt);
}
template <int N>
__device__ __forceinline__ uint32_t warp_kth_reg(const uint32_t (&key)[N], int kth, int nu) {
  uint32_t lo_and = 0xFFFFFFFFu, hi_or = 0u;
#pragma unroll
  for (int g = 0; g < N; g += 16) {
    if (g < nu) {
#pragma unroll
      for (int u = g; u < g + 16 && u < N; ++u) {
        if (key[u] != 0u) lo_and &= key[u];
        hi_or |= key[u];
      }
    }
  }
  lo_and = __reduce_and_sync(0xffffffffu, lo_and);
  hi_or = __reduce_or_sync(0xffffffffu, hi_or);
  const uint32_t diff = lo_and ^ hi_or;
  if (diff == 0u) return hi_or;                       // every present key is the same
  const int top = 31 - __clz(diff);
  uint32_t K = hi_or & ~((2u << top) - 1u);           // the bits above `top`, shared by all
  if (top == 31) K = 0u;
  for (int bit = top; bit >= 0; --bit) {
    const uint32_t c = K | (1u << bit);
    if (warp_count_ge(key, c, nu) >= (uint32_t)kth) K = c;
  }
  return K;
}
constexpr int kPThrPer = kPSampleTiles * kPM / 32;   // sampled scores per lane (64)

// Threshold key of query q: the score key of the r-th best visible sampled
// score, r = clamp(ceil(kPCandTarget * m / visible), 8, m) for m visible
// sampled entries. Queries with at most kCandCap visible entries get key 0
// (every visible entry is a candidate).
__global__ void __launch_bounds__(32 * kPSelWarps) k_prefill_threshold(const float* __restrict__ sample,
                                                                        int64_t n_samp, int tile_step,
                                                                        const int64_t* __restrict__ n_vis,
                                                                        int64_t n_keys, int Q,
                                                                        uint32_t* __restrict__ tau) {
  const int wq = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int q = blockIdx.x * kPSelWarps + wq;
  if (q >= Q) return;                           // warp-uniform; no block barrier below
  int64_t vis = n_vis ? n_vis[q] : n_keys;
  vis = vis < 0 ? 0 : (vis > n_keys ? n_keys : vis);
  if (vis <= kCandCap) {
    if (lane == 0) tau[q] = 0u;
    return;
  }
  const int64_t span = (int64_t)tile_step * kPM;
  int64_t m = 0;                                // visible sampled entries
  for (int64_t t = 0; t * kPM < n_samp; ++t) {
    const int64_t left = vis - t * span;
    m += left <= 0 ? 0 : (left < kPM ? left : kPM);
  }
  int64_t r = (kPCandTarget * m + vis - 1) / vis;
  r = r < 8 ? 8 : r;
  r = r > m ? m : r;
  uint32_t key[kPThrPer];
  const float* row = sample + (int64_t)q * n_samp;
#pragma unroll
  for (int u = 0; u < kPThrPer; ++u) {
    const int64_t j = lane + 32 * u;
    const int64_t entry = (j / kPM) * span + (j % kPM);
    key[u] = (j < n_samp && entry < vis) ? score_key(row[j]) : 0u;
  }
  const uint32_t K = warp_kth_reg(key, (int)r, kPThrPer);
  if (lane == 0) tau[q] = K;
}

// Bitonic sort, ascending, of 32 x 16 values held by a warp in registers:
// lane l holds elements l * 16 .. l * 16 + 15. Strides below 16 compare
// registers of one lane; larger strides exchange with lane l ^ (stride / 16).
__device__ __forceinline__ void warp_sort512(int32_t (&v)[16], int lane) {
#pragma unroll
  for (int size = 2; size <= 512; size <<= 1) {
#pragma unroll
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      if (stride >= 16) {
        const int m = stride >> 4;
        const bool lower = (lane & m) == 0;
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const int32_t o = __shfl_xor_sync(0xffffffffu, v[j], m);
          const bool up = ((lane * 16 + j) & size) == 0;
          v[j] = (lower == up) ? min(v[j], o) : max(v[j], o);
        }
      } else {
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          if (j & stride) continue;
          const bool up = ((lane * 16 + j) & size) == 0;
          const int32_t a = v[j], b = v[j | stride];
          if ((a > b) == up) { v[j] = b; v[j | stride] = a; }
        }
      }
    }
  }
}

// Exact Top-k of query q (one warp) over its candidate list; rows marked to
// be selected from their full score row are left to k_prefill_select_row.
// Writes the chosen positions ascending, then -1 up to k.
// Fast path (lists of up to 32 * kPSelLane slots, k <= 512): the score keys
// stay in registers and the need-th largest score key K comes from a warp
// bisection; when exactly `need` keys reach K, each lane reads the positions
// of its taken keys in one batch, the warp gathers them into registers and
// sorts them there. Otherwise (a long list, a large k, or a tie at K to be
// split by position, where the smallest positions win): the radix select
// over the list's full keys and a shared-memory sort.
constexpr int kPSelLane = 128;                     // list slots per lane on the fast path

struct ListSource {              // a query's candidate list (0 = a hole)
  const uint64_t* c;
  int n;
  __device__ bool get(int i, uint64_t& key) const { key = c[i]; return key != 0ull; }
};

__global__ void __launch_bounds__(32 * kPSelWarps, 1) k_prefill_select(const TopkHdr* __restrict__ hdr,
                                                                        const uint64_t* __restrict__ cand,
                                                                        const int64_t* __restrict__ n_vis,
                                                                        int64_t n_keys, int Q, int k,
                                                                        int32_t* __restrict__ idx) {
  __shared__ uint32_t h[kPSelWarps][kPSelBins];   // radix digits, then the chosen positions
  const int wq = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int q = blockIdx.x * kPSelWarps + wq;
  if (q >= Q || hdr[q].overflow != 0) return;     // warp-uniform; no block barrier below
  const uint32_t cnt_slots = hdr[q].cnt, holes = hdr[q].done;
  const int n = (int)min(cnt_slots, (uint32_t)kCandCap);
  const int valid = (int)(cnt_slots - holes);
  const int need = valid < k ? valid : k;
  const uint64_t* lst = cand + (int64_t)q * kCandCap;
  int32_t* sel = reinterpret_cast<int32_t*>(h[wq]);
  int32_t* out = idx + (int64_t)q * k;
  (void)n_vis;
  (void)n_keys;
  // fast path unless the list is long, k large, or a tie at the boundary
  // score has to be split by position
  bool general = n > 32 * kPSelLane || k > 512;
  const int nu = (n + 31) / 32;                    // register slots holding keys (warp-uniform)
  uint32_t hk[kPSelLane];
  uint32_t K = 1;                                  // every present key (holes are 0)
#pragma unroll
  for (int u = 0; u < kPSelLane; ++u) hk[u] = 0u;
  if (!general) {
#pragma unroll
    for (int g = 0; g < kPSelLane; g += 16) {
#pragma unroll
      for (int u = g; u < g + 16; ++u) {
        const int i = lane + 32 * u;
        if (g < nu && i < n) hk[u] = (uint32_t)(lst[i] >> 32);
      }
    }
    if (valid > need) {
      K = warp_kth_reg(hk, need, nu);
      general = warp_count_ge(hk, K, nu) != (uint32_t)need;
    }
  }
  if (general) {
    // general path: radix select, then a shared-memory bitonic sort
    ListSource src{lst, n};
    uint64_t thr = 1;
    if (valid > need) thr = warp_kth(src, need, false, h[wq], lane);
    __syncwarp();
    int cnt = 0;
    for (int i0 = 0; i0 < n; i0 += 32) {
      const int i = i0 + lane;
      uint64_t key = 0;
      const bool t = i < n && src.get(i, key) && key >= thr;
      const uint32_t bal = __ballot_sync(0xffffffffu, t);
      if (t) {
        const int at = cnt + __popc(bal & ((1u << lane) - 1u));
        if (at < need) sel[at] = cand_pos_of(key);
      }
      cnt += __popc(bal);
    }
    int np = 1;
    while (np < need) np <<= 1;
    for (int i = need + lane; i < np; i += 32) sel[i] = 0x7FFFFFFF;
    __syncwarp();
    for (int size = 2; size <= np; size <<= 1) {
      for (int stride = size >> 1; stride > 0; stride >>= 1) {
        for (int i = lane; i < np / 2; i += 32) {
          const int lo = 2 * i - (i & (stride - 1));
          const int hi = lo + stride;
          const bool up = (lo & size) == 0;
          const int32_t x = sel[lo], y = sel[hi];
          if ((x > y) == up) { sel[lo] = y; sel[hi] = x; }
        }
        __syncwarp();
      }
    }
    for (int i = lane; i < k; i += 32) out[i] = i < need ? sel[i] : -1;
    return;
  }
  // this lane's taken slots, their place in the warp's list, their positions
  uint32_t mine = 0;
#pragma unroll
  for (int g = 0; g < kPSelLane; g += 16) {
    if (g < nu) {
#pragma unroll
      for (int u = g; u < g + 16; ++u) {
        mine += hk[u] >= K ? 1u : 0u;
      }
    }
  }
  uint32_t incl = mine;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const uint32_t o = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += o;
  }
  uint32_t at = incl - mine;
#pragma unroll
  for (int g = 0; g < kPSelLane; g += 16) {
    if (g < nu) {
#pragma unroll
      for (int u = g; u < g + 16; ++u) {
        if (hk[u] >= K) {
          if (at < (uint32_t)need) sel[at] = cand_pos_of(lst[lane + 32 * u]);
          ++at;
        }
      }
    }
  }
  __syncwarp();
  int32_t v[16];
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    const int e = lane * 16 + j;
    v[j] = e < need ? sel[e] : 0x7FFFFFFF;
  }
  warp_sort512(v, lane);
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    const int e = lane * 16 + j;
    if (e < k) out[e] = e < need ? v[j] : -1;
  }
}

// Exact Top-k of each marked query (one warp) from its full score row
// (stride n_keys): radix select over the row, positions ascending, then -1
// up to k. Unmarked queries return at once.
__global__ void __launch_bounds__(32 * kPSelWarps) k_prefill_select_row(const TopkHdr* __restrict__ hdr,
                                                                         const float* __restrict__ scores,
                                                                         const int64_t* __restrict__ n_vis,
                                                                         int64_t n_keys, int Q, int k,
                                                                         int32_t* __restrict__ idx) {
  __shared__ uint32_t h[kPSelWarps][kPSelBins];   // radix digits, then the chosen positions
  const int wq = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int q = blockIdx.x * kPSelWarps + wq;
  if (q >= Q || hdr[q].overflow == 0) return;     // warp-uniform; no block barrier below
  int64_t vis = n_vis ? n_vis[q] : n_keys;
  vis = vis < 0 ? 0 : (vis > n_keys ? n_keys : vis);
  const int n = (int)vis;
  const int need = n < k ? n : k;
  int32_t* sel = reinterpret_cast<int32_t*>(h[wq]);
  RowSource src{scores + (int64_t)q * n_keys, n};
  uint64_t thr = 1;
  if (n > need) thr = warp_kth(src, need, false, h[wq], lane);
  __syncwarp();
  int cnt = 0;
  for (int i0 = 0; i0 < n; i0 += 32) {
    const int i = i0 + lane;
    uint64_t key = 0;
    const bool t = i < n && src.get(i, key) && key >= thr;
    const uint32_t bal = __ballot_sync(0xffffffffu, t);
    if (t) {
      const int at = cnt + __popc(bal & ((1u << lane) - 1u));
      if (at < need) sel[at] = cand_pos_of(key);
    }
    cnt += __popc(bal);
  }
  int np = 1;
  while (np < need) np <<= 1;
  for (int i = need + lane; i < np; i += 32) sel[i] = 0x7FFFFFFF;
  __syncwarp();
  for (int size = 2; size <= np; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      for (int i = lane; i < np / 2; i += 32) {
        const int lo = 2 * i - (i & (stride - 1));
        const int hi = lo + stride;
        const bool up = (lo & size) == 0;
        const int32_t x = sel[lo], y = sel[hi];
        if ((x > y) == up) { sel[lo] = y; sel[hi] = x; }
      }
      __syncwarp();
    }
  }
  int32_t* out = idx + (int64_t)q * k;
  for (int i = lane; i < k; i += 32) out[i] = i < need ? sel[i] : -1;
}

// A query whose candidate list cannot hold its Top-k exactly (fewer than
// min(k, visible) candidates, or more than kCandCap) takes the Top-K's slow
// path over its full score row; its query tile is marked for the full write.
__global__ void k_prefill_check(TopkHdr* __restrict__ hdr, const int64_t* __restrict__ n_vis, int64_t n_keys,
                                int Q, int k, int32_t* __restrict__ gate) {
  const int q = blockIdx.x * blockDim.x + threadIdx.x;
  if (q >= Q) return;
  int64_t vis = n_vis ? n_vis[q] : n_keys;
  vis = vis < 0 ? 0 : (vis > n_keys ? n_keys : vis);
  const int64_t need = vis < k ? vis : k;
  const uint32_t cnt = hdr[q].cnt;                 // slots reserved (filled or holes)
  const uint32_t real = cnt - hdr[q].done;          // slots filled
  const bool ov = cnt > (uint32_t)kCandCap || (int64_t)real < need;
  hdr[q].overflow = ov ? 1u : 0u;
  if (ov) gate[q / kPQ] = 1;
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
  if (cudaFuncSetAttribute(k_prefill_index<kPWrite>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           PrefillSmem::kBytes) != cudaSuccess ||
      cudaFuncSetAttribute(k_prefill_index<kPFilter>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           PrefillSmem::kBytes) != cudaSuccess)
    return CSA2_ERR_CUDA;
  return CSA2_OK;
}

// One pass over every query tile, in launches of at most kPMaxQTiles tiles.
static int run_pass(const CUtensorMap& mk, const CUtensorMap& mq, PrefillPass p, cudaStream_t s) {
  const int qtiles_all = (p.Q + kPQ - 1) / kPQ;
  p.wait_ns = debug_wait_ns();
  p.fault = debug_fault() == kFaultPrefill ? 1 : 0;
  for (int qt0 = 0; qt0 < qtiles_all; qt0 += kPMaxQTiles) {
    p.qt0 = qt0;
    p.qtiles = qtiles_all - qt0 < kPMaxQTiles ? qtiles_all - qt0 : kPMaxQTiles;
    const int64_t units = (int64_t)p.qtiles * p.seq_tiles;
    const unsigned grid = (unsigned)(units < kSMs ? units : kSMs);
    if (p.mode == kPFilter)
      k_prefill_index<kPFilter><<<grid, kPThreads, PrefillSmem::kBytes, s>>>(mk, mq, p);
    else
      k_prefill_index<kPWrite><<<grid, kPThreads, PrefillSmem::kBytes, s>>>(mk, mq, p);
    count_launch();
    const int rc = launch_status();
    if (rc != CSA2_OK) return rc;
  }
  return CSA2_OK;
}

static int make_maps(CUtensorMap* mk, CUtensorMap* mq, const uint8_t* qI, int Q, const uint8_t* kI,
                     int64_t n_keys) {
  if (!make_tmap_rows128(mk, kI, (uint64_t)n_keys, kPK, kPM)) return CSA2_ERR_INVALID_ARG;
  if (!make_tmap_rows128(mq, qI, (uint64_t)Q * kPH, kPK, kPN)) return CSA2_ERR_INVALID_ARG;
  return CSA2_OK;
}

static PrefillPass pass_base(const float* w, int Q, int64_t n_keys, int32_t* st) {
  PrefillPass p{};
  p.w = w;
  p.Q = Q;
  p.n_keys = n_keys;
  p.st = st;
  p.tile_step = 1;
  p.seq_tiles = (n_keys + kPM - 1) / kPM;
  p.mode = kPWrite;
  return p;
}

// Every score: scores[q * stride + j] for j < n_keys.
int launch_prefill_index(const uint8_t* qI, const float* w, int Q, const uint8_t* kI, int64_t n_keys, float* scores,
                         int64_t stride, int32_t* st, cudaStream_t s) {
  if (Q == 0 || n_keys == 0) return CSA2_OK;
  CUtensorMap mk, mq;
  int rc = make_maps(&mk, &mq, qI, Q, kI, n_keys);
  if (rc != CSA2_OK) return rc;
  PrefillPass p = pass_base(w, Q, n_keys, st);
  p.scores = scores;
  p.stride = stride;
  return run_pass(mk, mq, p, s);
}

// Sampling geometry: every S-th entry tile, at most kPSampleTiles of them.
static void sample_geometry(int64_t n_keys, int* S, int64_t* seq_tiles) {
  const int64_t ktiles = (n_keys + kPM - 1) / kPM;
  int64_t st = (ktiles + kPSampleTiles - 1) / kPSampleTiles;
  if (st < kPSampleMin) st = kPSampleMin;
  *S = (int)st;
  *seq_tiles = (ktiles + st - 1) / st;
}

size_t prefill_select_ws_bytes(int Q, int64_t n_keys) {
  int S;
  int64_t seq;
  sample_geometry(n_keys, &S, &seq);
  const size_t qtiles = (size_t)(Q + kPQ - 1) / kPQ;
  return align256((size_t)Q * (size_t)seq * kPM * 4) + align256((size_t)Q * 4) + align256(qtiles * 4);
}

// Steps 1-3: the candidates of every query (into the Top-K workspace tk).
int launch_prefill_candidates(const uint8_t* qI, const float* w, int Q, const uint8_t* kI, int64_t n_keys,
                              const int64_t* n_vis, void* tk, void* sel_ws, int32_t* st, cudaStream_t s) {
  if (Q == 0) return CSA2_OK;
  int rc = topk_prepare(tk, Q, s);
  if (rc != CSA2_OK) return rc;
  int S;
  int64_t seq;
  sample_geometry(n_keys, &S, &seq);
  char* p8 = static_cast<char*>(sel_ws);
  float* sample = reinterpret_cast<float*>(p8);
  p8 += align256((size_t)Q * (size_t)seq * kPM * 4);
  uint32_t* tau = reinterpret_cast<uint32_t*>(p8);
  p8 += align256((size_t)Q * 4);
  int32_t* gate = reinterpret_cast<int32_t*>(p8);
  if (cudaMemsetAsync(gate, 0, (size_t)((Q + kPQ - 1) / kPQ) * 4, s) != cudaSuccess) return CSA2_ERR_CUDA;
  if (n_keys == 0) return CSA2_OK;
  CUtensorMap mk, mq;
  if ((rc = make_maps(&mk, &mq, qI, Q, kI, n_keys)) != CSA2_OK) return rc;
  if (n_keys > kCandCap) {                        // shorter rows take every visible entry
    PrefillPass p = pass_base(w, Q, n_keys, st);
    p.n_vis = n_vis;
    p.scores = sample;
    p.stride = seq * kPM;
    p.tile_step = S;
    p.seq_tiles = seq;
    if ((rc = run_pass(mk, mq, p, s)) != CSA2_OK) return rc;
  }
  k_prefill_threshold<<<(Q + kPSelWarps - 1) / kPSelWarps, 32 * kPSelWarps, 0, s>>>(sample, seq * kPM, S, n_vis,
                                                                                    n_keys, Q, tau);
  count_launch();
  if ((rc = launch_status()) != CSA2_OK) return rc;
  PrefillPass p = pass_base(w, Q, n_keys, st);
  p.n_vis = n_vis;
  p.mode = kPFilter;
  p.tau = tau;
  p.hdr = topk_ws_hdr(tk, Q);
  p.cand = topk_ws_cand(tk, Q);
  return run_pass(mk, mq, p, s);
}

// Steps 4-5: mark the queries the candidates cannot serve, write the full
// rows of their query tiles into `scores` (stride n_keys), select.
int launch_prefill_finish(const uint8_t* qI, const float* w, int Q, const uint8_t* kI, int64_t n_keys,
                          const int64_t* n_vis, int k, int32_t* idx, float* scores, void* tk, void* sel_ws,
                          int32_t* st, cudaStream_t s) {
  if (Q == 0) return CSA2_OK;
  int S;
  int64_t seq;
  sample_geometry(n_keys, &S, &seq);
  char* p8 = static_cast<char*>(sel_ws) + align256((size_t)Q * (size_t)seq * kPM * 4) + align256((size_t)Q * 4);
  int32_t* gate = reinterpret_cast<int32_t*>(p8);
  int rc;
  k_prefill_check<<<(Q + 255) / 256, 256, 0, s>>>(topk_ws_hdr(tk, Q), n_vis, n_keys, Q, k, gate);
  count_launch();
  if ((rc = launch_status()) != CSA2_OK) return rc;
  if (n_keys > 0) {
    CUtensorMap mk, mq;
    if ((rc = make_maps(&mk, &mq, qI, Q, kI, n_keys)) != CSA2_OK) return rc;
    PrefillPass p = pass_base(w, Q, n_keys, st);
    p.n_vis = n_vis;
    p.gate = gate;
    p.scores = scores;
    p.stride = n_keys;
    if ((rc = run_pass(mk, mq, p, s)) != CSA2_OK) return rc;
  }
  k_prefill_select<<<(Q + kPSelWarps - 1) / kPSelWarps, 32 * kPSelWarps, 0, s>>>(
      topk_ws_hdr(tk, Q), topk_ws_cand(tk, Q), n_vis, n_keys, Q, k, idx);
  count_launch();
  if ((rc = launch_status()) != CSA2_OK) return rc;
  k_prefill_select_row<<<(Q + kPSelWarps - 1) / kPSelWarps, 32 * kPSelWarps, 0, s>>>(topk_ws_hdr(tk, Q), scores,
                                                                                     n_vis, n_keys, Q, k, idx);
  count_launch();
  return launch_status();
}

}  // namespace csa2
