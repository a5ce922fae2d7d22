// topk.cu — deterministic Top-K selection for the CSA2 indexer.
//
// [CSA2] wire.sakhanda.co, "DeepSeek AI выпустила DeepSeek-V4.1-Flash ...",
//        section "Сжатое разреженное внимание 2 (CSA2)": Full selects new
//        Top-512 indices; Reindex selects again among the pool; the pool
//        itself keeps the best 2048 blocks.
//
// Order: score descending, then position ascending. Each candidate becomes
// a unique 64-bit key (order-preserving score bits << 32 | ~position), so the
// k best are exactly the k largest keys and the result does not depend on
// the order in which threads or CTAs visit the candidates.
//
// Pipeline per row:
//   1. histogram of the 12 high score-key bits (4096 bins) over the row,
//      fused into the indexer scan when the scan runs just before; the last
//      CTA of the row finds the threshold bin (the one holding the k-th
//      largest score) and flags the row if more than kCandCap entries lie at
//      or above it;
//   2. rows longer than kDirectRows: ordered compaction. The row is cut into
//      chunks of kChunk entries; a CTA compacts a chunk (the entries at or
//      above the threshold bin, in index order), reserves room for it with a
//      single atomic and records (base, count) in the row's chunk table;
//   3. one CTA per row (512 threads for k <= 512, 1024 above) gathers the
//      candidates in index order (through the
//      chunk table, or straight from the row when it is short). When the
//      positions increase with the index (position-indexed rows, pool slots)
//      the k-th score is resolved inside the threshold bin by two 10-bit
//      histogram passes, ties at that score go to the first entries in index
//      order (the smallest positions), and the chosen entries are written in
//      index order, which is ascending position order: no sort. Otherwise,
//      and for flagged rows (over the whole row in global memory), an exact
//      radix select over the 64-bit keys is followed by a sort.
#include "common.cuh"

namespace csa2 {


constexpr int kChunk = kTkThreads * 8;        // entries per compaction chunk
constexpr int kMaxChunks = 4096;              // chunk-table entries per row (rows up to 8M entries)
constexpr int64_t kDirectRows = 32768;        // rows this short skip step 2

// Workspace layout (all offsets 256-byte aligned):
//   hist [B][kHistBins] u32 | hdr [B] TopkHdr | cand [B][kCandCap] u64 |
//   tab [B][kMaxChunks] {base, count}
static size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }
size_t topk_ws_bytes(int B) {
  return align256((size_t)B * kHistBins * 4) + align256((size_t)B * sizeof(TopkHdr)) +
         align256((size_t)B * kCandCap * 8) + align256((size_t)B * kMaxChunks * 8);
}
struct TopkWs {
  uint32_t* hist;
  TopkHdr* hdr;
  uint64_t* cand;
  uint2* tab;
};
static TopkWs topk_ws(void* ws, int B) {
  char* p = static_cast<char*>(ws);
  TopkWs r;
  r.hist = reinterpret_cast<uint32_t*>(p);
  p += align256((size_t)B * kHistBins * 4);
  r.hdr = reinterpret_cast<TopkHdr*>(p);
  p += align256((size_t)B * sizeof(TopkHdr));
  r.cand = reinterpret_cast<uint64_t*>(p);
  p += align256((size_t)B * kCandCap * 8);
  r.tab = reinterpret_cast<uint2*>(p);
  return r;
}
uint32_t* topk_ws_hist(void* ws) { return static_cast<uint32_t*>(ws); }
TopkHdr* topk_ws_hdr(void* ws, int B) { return topk_ws(ws, B).hdr; }
uint64_t* topk_ws_cand(void* ws, int B) { return topk_ws(ws, B).cand; }


// Candidates of row b: the first ceil(n[b] / len_div) entries, at most n_max
// (n == NULL: every row has n_max entries).
__device__ __forceinline__ int64_t row_len(const int64_t* n, int b, int len_div, int64_t n_max) {
  if (n == nullptr) return n_max;
  int64_t v = n[b];
  v = v <= 0 ? 0 : (v + len_div - 1) / len_div;
  return v < n_max ? v : n_max;
}

// Exclusive prefix sum of one value per thread over a CTA of NT threads;
// *total receives the CTA's sum. s_warp holds NT / 32 words. Contains two
// barriers, so every thread of the CTA must call it.
template <int NT>
__device__ __forceinline__ uint32_t block_excl_scan(uint32_t v, uint32_t* s_warp, uint32_t* total) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  uint32_t incl = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const uint32_t t = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += t;
  }
  if (lane == 31) s_warp[wid] = incl;
  __syncthreads();
  uint32_t before = 0, tot = 0;
#pragma unroll
  for (int w = 0; w < NT / 32; ++w) {
    const uint32_t x = s_warp[w];
    before += w < wid ? x : 0u;
    tot += x;
  }
  __syncthreads();
  *total = tot;
  return before + incl - v;
}

// Eight consecutive entries i..i+7 of a row (fewer at its end): score and
// position (-1 = absent), with vector loads when the whole group is inside the
// row and 16-byte aligned.
__device__ __forceinline__ void load8(const float* __restrict__ s, const int32_t* __restrict__ cp, int64_t i,
                                      int64_t len, float* v, int32_t* p) {
  const bool vec = i + 8 <= len &&
                   ((reinterpret_cast<uintptr_t>(s + i) | (cp ? reinterpret_cast<uintptr_t>(cp + i) : 0)) & 15) == 0;
  if (vec) {
    const float4 a = *reinterpret_cast<const float4*>(s + i), c = *reinterpret_cast<const float4*>(s + i + 4);
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = c.x; v[5] = c.y; v[6] = c.z; v[7] = c.w;
    if (cp) {
      const int4 pa = *reinterpret_cast<const int4*>(cp + i), pb = *reinterpret_cast<const int4*>(cp + i + 4);
      p[0] = pa.x; p[1] = pa.y; p[2] = pa.z; p[3] = pa.w; p[4] = pb.x; p[5] = pb.y; p[6] = pb.z; p[7] = pb.w;
    } else {
#pragma unroll
      for (int u = 0; u < 8; ++u) p[u] = (int32_t)(i + u);
    }
  } else {
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const bool in = i + u < len;
      v[u] = in ? s[i + u] : 0.f;
      p[u] = in ? (cp ? cp[i + u] : (int32_t)(i + u)) : -1;
    }
  }
}

// ---- step 1 (standalone form) --------------------------------------------
__global__ void __launch_bounds__(kTkThreads) k_topk_hist(const float* __restrict__ scores,
                                                          const int32_t* __restrict__ cand_pos,
                                                          int64_t stride, const int64_t* __restrict__ n,
                                                          int len_div, int64_t n_max, int64_t per,
                                                          uint32_t* __restrict__ hist, TopkHdr* __restrict__ hdr,
                                                          int k) {
  __shared__ uint32_t sh[kHistBins];
  const int b = blockIdx.y;
  for (int i = threadIdx.x; i < kHistBins; i += kTkThreads) sh[i] = 0;
  pdl_trigger();
  pdl_wait();
  __syncthreads();
  const int64_t nb = row_len(n, b, len_div, n_max);
  const int64_t c0 = (int64_t)blockIdx.x * per, c1 = min(c0 + per, nb);
  const float* s = scores + (int64_t)b * stride;
  const int32_t* cp = cand_pos ? cand_pos + (int64_t)b * stride : nullptr;
  for (int64_t i = c0 + threadIdx.x; i < c1; i += kTkThreads) {
    if (cp && cp[i] < 0) continue;
    atomicAdd(&sh[score_key(s[i]) >> 20], 1u);
  }
  topk_hist_flush(sh, hist + (int64_t)b * kHistBins, hdr + b, k, gridDim.x);
}

// ---- step 2 ----------------------------------------------------------------
// Ordered compaction of rows longer than kDirectRows: chunk c of row b holds
// entries [c * kChunk, (c + 1) * kChunk); thread t owns eight consecutive
// entries of it. The chunk's candidates land contiguously, in index order, at
// a base reserved by one atomic, and tab[b][c] = (base, count).
__global__ void __launch_bounds__(kTkThreads) k_topk_compact(const float* __restrict__ scores,
                                                             const int32_t* __restrict__ cand_pos,
                                                             int64_t stride, const int64_t* __restrict__ n,
                                                             int len_div, int64_t n_max,
                                                             TopkHdr* __restrict__ hdr,
                                                             uint64_t* __restrict__ cand, uint2* __restrict__ tab) {
  __shared__ uint32_t s_warp[kTkThreads / 32];
  __shared__ uint32_t s_base;
  pdl_trigger();
  pdl_wait();
  const int b = blockIdx.y;
  if (hdr[b].overflow) return;
  const int vbin = hdr[b].vbin;
  const int64_t nb = row_len(n, b, len_div, n_max);
  const int64_t nch = (nb + kChunk - 1) / kChunk;
  const float* s = scores + (int64_t)b * stride;
  const int32_t* cp = cand_pos ? cand_pos + (int64_t)b * stride : nullptr;
  uint64_t* out = cand + (int64_t)b * kCandCap;
  for (int64_t ch = blockIdx.x; ch < nch; ch += gridDim.x) {
    const int64_t i = ch * kChunk + (int64_t)threadIdx.x * 8;
    float v[8];
    int32_t p[8];
    load8(s, cp, i, nb, v, p);
    uint32_t take = 0;
#pragma unroll
    for (int u = 0; u < 8; ++u)
      if (p[u] >= 0 && (int)(score_key(v[u]) >> 20) >= vbin) take |= 1u << u;
    uint32_t tot;
    const uint32_t excl = block_excl_scan<kTkThreads>(__popc(take), s_warp, &tot);
    if (threadIdx.x == 0) {
      s_base = tot ? atomicAdd(&hdr[b].cnt, tot) : 0u;
      if (ch < kMaxChunks) tab[(int64_t)b * kMaxChunks + ch] = make_uint2(s_base, tot);
    }
    __syncthreads();
    uint32_t slot = s_base + excl;
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      if (!((take >> u) & 1)) continue;
      if (slot < (uint32_t)kCandCap) out[slot] = cand_key(v[u], p[u]);   // always: the row did not overflow
      ++slot;
    }
  }
}

// ---- step 3 ----------------------------------------------------------------
// The final kernel runs NT threads per row: 512 for k <= 512 (shorter
// barriers; measured faster), 1024 for larger k (the pool's 2048).
constexpr int kFinThreadsSmallK = 512, kFinThreadsLargeK = 1024;

// Key sources for the radix select.
struct SmemKeys {
  const uint64_t* keys;
  int cnt;
  __device__ int64_t size() const { return cnt; }
  __device__ bool get(int64_t i, uint64_t& key) const { key = keys[i]; return true; }
};
struct RowKeys {
  const float* s;
  const int32_t* cp;
  int64_t cnt;
  __device__ int64_t size() const { return cnt; }
  __device__ bool get(int64_t i, uint64_t& key) const {
    const int32_t p = cp ? cp[i] : (int32_t)i;
    if (p < 0) return false;
    key = cand_key(s[i], p);
    return true;
  }
};

// Exact key of the k-th largest among the source's keys (all distinct);
// requires at least k keys. MSD radix, 8 bits per pass.
template <int NT, class Src>
__device__ uint64_t radix_kth(const Src& src, int k, uint32_t* h256) {
  __shared__ uint64_t s_prefix;
  __shared__ int s_remaining;
  __shared__ unsigned long long s_and, s_or;
  const int tid = threadIdx.x;
  // bits shared by every key are fixed: skip the digits above the first difference
  if (tid == 0) { s_and = ~0ull; s_or = 0ull; }
  __syncthreads();
  {
    unsigned long long a = ~0ull, o = 0ull;
    const int64_t m = src.size();
    for (int64_t i = tid; i < m; i += NT) {
      uint64_t key;
      if (src.get(i, key)) { a &= key; o |= key; }
    }
    for (int off = 16; off > 0; off >>= 1) {
      a &= __shfl_xor_sync(0xffffffffu, a, off);
      o |= __shfl_xor_sync(0xffffffffu, o, off);
    }
    if ((tid & 31) == 0) { atomicAnd(&s_and, a); atomicOr(&s_or, o); }
  }
  __syncthreads();
  const uint64_t diff = s_and ^ s_or;                 // bits that are not common to all keys
  const int top = diff ? 63 - __clzll((long long)diff) : -1;
  int start = 56;
  while (start > 0 && start > top) start -= 8;        // first digit holding a differing bit
  uint64_t mask = start < 56 ? ~((1ull << (start + 8)) - 1) : 0ull;
  uint64_t prefix = s_and & mask;
  int remaining = k;
  for (int shift = start; shift >= 0; shift -= 8) {
    for (int i = tid; i < 256; i += NT) h256[i] = 0;
    __syncthreads();
    const int64_t m = src.size();
    const int lane = tid & 31;
    for (int64_t i0 = 0; i0 < m; i0 += NT) {
      const int64_t i = i0 + tid;
      uint64_t key = 0;
      const bool ok = i < m && src.get(i, key) && (key & mask) == prefix;
      const uint32_t dgt = ok ? (uint32_t)((key >> shift) & 255) : 256u;
      const uint32_t peers = __match_any_sync(0xffffffffu, dgt);   // lanes holding the same digit
      if (ok && lane == __ffs(peers) - 1) atomicAdd(&h256[dgt], (uint32_t)__popc(peers));
    }
    __syncthreads();
    if (tid < 32) {
      // lane l owns digits [255-8l-7, 255-8l], counted from the top
      uint32_t loc = 0;
      for (int j = 0; j < 8; ++j) loc += h256[255 - 8 * tid - j];
      uint32_t incl = loc;
      for (int off = 1; off < 32; off <<= 1) {
        const uint32_t v = __shfl_up_sync(0xffffffffu, incl, off);
        if (tid >= off) incl += v;
      }
      const uint32_t excl = incl - loc;
      if (excl < (uint32_t)remaining && incl >= (uint32_t)remaining) {
        uint32_t run = excl;
        for (int j = 0; j < 8; ++j) {
          const int dgt = 255 - 8 * tid - j;
          const uint32_t c = h256[dgt];
          if (run + c >= (uint32_t)remaining) {
            s_prefix = prefix | ((uint64_t)dgt << shift);
            s_remaining = remaining - (int)run;
            break;
          }
          run += c;
        }
      }
    }
    __syncthreads();
    prefix = s_prefix;
    remaining = s_remaining;
    mask |= (uint64_t)255 << shift;
    __syncthreads();
  }
  return prefix;
}

// Bitonic sort of sel[0..np) ascending (np a power of two, padded with INT_MAX).
template <int NT>
__device__ void bitonic_sort_i32(int32_t* sel, int np) {
  for (int size = 2; size <= np; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      __syncthreads();
      for (int i = threadIdx.x; i < np / 2; i += NT) {
        const int lo = 2 * i - (i & (stride - 1));
        const int hi = lo + stride;
        const bool up = ((lo & size) == 0);
        const int32_t a = sel[lo], c = sel[hi];
        if ((a > c) == up) { sel[lo] = c; sel[hi] = a; }
      }
    }
  }
  __syncthreads();
}

template <int NT, class Src>
__device__ void select_and_write(const Src& src, int k, int64_t n_keys, int32_t* __restrict__ out,
                                 uint32_t* h256, int32_t* sel) {
  __shared__ uint32_t s_cnt;
  const int tid = threadIdx.x;
  uint64_t thr = 0;
  if (n_keys > k) thr = radix_kth<NT>(src, k, h256);
  if (tid == 0) s_cnt = 0;
  __syncthreads();
  const int64_t m = src.size();
  const int lane = tid & 31;
  for (int64_t i0 = 0; i0 < m; i0 += NT) {
    const int64_t i = i0 + tid;
    uint64_t key = 0;
    const bool take = i < m && src.get(i, key) && key >= thr;
    const uint32_t bal = __ballot_sync(0xffffffffu, take);
    uint32_t base = 0;
    if (bal) {
      if (lane == __ffs(bal) - 1) base = atomicAdd(&s_cnt, (uint32_t)__popc(bal));
      base = __shfl_sync(0xffffffffu, base, __ffs(bal) - 1);
    }
    if (take) {
      const uint32_t slot = base + __popc(bal & ((1u << lane) - 1u));
      if (slot < (uint32_t)k) sel[slot] = cand_pos_of(key);
    }
  }
  __syncthreads();
  const int cnt = (int)min(s_cnt, (uint32_t)k);
  if (k <= 512) {
    // ascending order by rank: the chosen positions are distinct, so the rank
    // of one is the number of chosen positions below it (reads broadcast)
    for (int i = tid; i < cnt; i += NT) {
      const int32_t mine = sel[i];
      int rank = 0;
      for (int j = 0; j < cnt; ++j) rank += sel[j] < mine;
      out[rank] = mine;
    }
    for (int i = cnt + tid; i < k; i += NT) out[i] = -1;
  } else {
    int np = 1;
    while (np < k) np <<= 1;
    for (int i = cnt + tid; i < np; i += NT) sel[i] = 0x7FFFFFFF;
    bitonic_sort_i32<NT>(sel, np);
    for (int i = tid; i < k; i += NT) out[i] = i < cnt ? sel[i] : -1;
  }
}

// Digit d of a 1024-bin histogram at which the count taken from the top
// reaches `need` (> 0, at most the histogram's sum), found by one warp: lane l
// sums bins 1023 - 32 l - i (i < 32, read in a rotated order so the lanes hit
// distinct banks), a warp scan picks the lane, and a second scan over that
// lane's bins picks the digit. *digit = d and *above = the count in bins
// above d (both 0 for an inconsistent histogram).
__device__ void warp_digit_from_top(const uint32_t* h, uint32_t need, int* digit, uint32_t* above) {
  const int lane = threadIdx.x & 31;
  // row j (from the top) holds digits 1023 - 32 j - i, i = 0..31; lane l
  // reads element l of every row (consecutive words: conflict-free), the 32
  // loads independent, and each row's total is one warp reduction
  uint32_t row_tot = 0;                                // lane j: the total of row j
#pragma unroll
  for (int j = 0; j < 32; ++j) {
    const uint32_t t = __reduce_add_sync(0xffffffffu, h[1023 - 32 * j - lane]);
    if (lane == j) row_tot = t;
  }
  uint32_t incl = row_tot;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const uint32_t t = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += t;
  }
  const uint32_t excl = incl - row_tot;
  const uint32_t hit = __ballot_sync(0xffffffffu, excl < need && incl >= need);
  *digit = 0;
  *above = 0;
  if (!hit) return;
  const int L = __ffs(hit) - 1;
  const uint32_t base = __shfl_sync(0xffffffffu, excl, L);
  const uint32_t c = h[1023 - 32 * L - lane];
  uint32_t inc2 = c;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const uint32_t t = __shfl_up_sync(0xffffffffu, inc2, off);
    if (lane >= off) inc2 += t;
  }
  const uint32_t ex2 = base + inc2 - c;
  const uint32_t hit2 = __ballot_sync(0xffffffffu, ex2 < need && ex2 + c >= need);
  if (!hit2) return;
  const int i = __ffs(hit2) - 1;
  *digit = 1023 - 32 * L - i;
  *above = __shfl_sync(0xffffffffu, ex2, i);
}

// Candidates keys[0..cnt) in index order with increasing positions, all at or
// above threshold bin vbin: write the k best positions, ascending, to out.
// h1, h2: two 1024-entry shared histograms; s_warp: the block scan's scratch.
template <int NT>
__device__ void ordered_select(const uint64_t* keys, int cnt, int vbin, int k, int32_t* __restrict__ out,
                               uint32_t* h1, uint32_t* h2, uint32_t* s_warp) {
  __shared__ uint32_t s_above, s_aA, s_aB;
  __shared__ int s_dA, s_dB;
  const int tid = threadIdx.x, lane = tid & 31;
  if (cnt <= k) {
    for (int i = tid; i < k; i += NT) out[i] = i < cnt ? cand_pos_of(keys[i]) : -1;
    return;
  }
  for (int i = tid; i < 1024; i += NT) {
    h1[i] = 0;
    h2[i] = 0;
  }
  if (tid == 0) s_above = 0;
  __syncthreads();
  // entries above the threshold bin are all taken; score-key bits 19..10 of
  // the entries in it
  uint32_t above = 0;
  for (int i = tid; i < cnt; i += NT) {
    const uint64_t key = keys[i];
    const int bin = (int)(key >> 52);
    if (bin > vbin) ++above;
    else if (bin == vbin) atomicAdd(&h1[(key >> 42) & 1023], 1u);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) above += __shfl_xor_sync(0xffffffffu, above, off);
  if (lane == 0 && above) atomicAdd(&s_above, above);
  __syncthreads();
  if (tid < 32) {                                      // the k-th score lies in the bin: need >= 1
    int d;
    uint32_t a;
    warp_digit_from_top(h1, (uint32_t)k - s_above, &d, &a);
    if (lane == 0) { s_dA = d; s_aA = a; }
  }
  __syncthreads();
  const uint32_t need = (uint32_t)k - s_above - s_aA;
  const uint64_t preA = ((uint64_t)vbin << 10) | (uint64_t)s_dA;   // score key >> 10
  // score-key bits 9..0 of the entries sharing that prefix
  for (int i = tid; i < cnt; i += NT) {
    const uint64_t key = keys[i];
    if ((key >> 42) == preA) atomicAdd(&h2[(key >> 32) & 1023], 1u);
  }
  __syncthreads();
  if (tid < 32) {
    int d;
    uint32_t a;
    warp_digit_from_top(h2, need, &d, &a);
    if (lane == 0) { s_dB = d; s_aB = a; }
  }
  __syncthreads();
  const uint32_t r = need - s_aB;                      // entries to take at exactly the k-th score
  const uint32_t thr = (uint32_t)((preA << 10) | (uint64_t)s_dB);
  // ordered output: thread t owns entries [lo, hi). One scan of the packed
  // counts (strictly above | ties << 16; both < 2^16) gives both prefixes:
  // the entry's slot is (above before it) + min(ties before it, r), as ties
  // at thr go to the first r in index order.
  const int S = (cnt + NT - 1) / NT;
  const int lo = min(tid * S, cnt), hi = min(lo + S, cnt);
  uint32_t gt = 0, ties = 0;
  for (int i = lo; i < hi; ++i) {
    const uint32_t sk = (uint32_t)(keys[i] >> 32);
    gt += sk > thr;
    ties += sk == thr;
  }
  uint32_t tot;
  const uint32_t pre = block_excl_scan<NT>(gt | (ties << 16), s_warp, &tot);
  uint32_t tr = pre >> 16;
  uint32_t o = (pre & 0xFFFFu) + min(tr, r);
  for (int i = lo; i < hi; ++i) {
    const uint32_t sk = (uint32_t)(keys[i] >> 32);
    bool take = sk > thr;
    if (sk == thr) take = tr++ < r;
    if (take && o < (uint32_t)k) out[o++] = cand_pos_of(keys[i]);
  }
}

// Gather modes of step 3.
enum FinalMode : int { kFinDirect = 0, kFinTable = 1, kFinUnordered = 2 };

template <int NT>
__global__ void __launch_bounds__(NT) k_topk_final(const float* __restrict__ scores,
                                                            const int32_t* __restrict__ cand_pos,
                                                            int64_t stride, const int64_t* __restrict__ n,
                                                            int len_div, int64_t n_max, int k,
                                                            const TopkHdr* __restrict__ hdr,
                                                            const uint64_t* __restrict__ cand,
                                                            const uint2* __restrict__ tab, int mode,
                                                            int32_t* __restrict__ idx_out) {
  extern __shared__ __align__(16) unsigned char smem[];
  uint64_t* keys = reinterpret_cast<uint64_t*>(smem);                 // kCandCap
  uint32_t* h = reinterpret_cast<uint32_t*>(keys + kCandCap);         // 1024 (256 for the radix select)
  int32_t* sel = reinterpret_cast<int32_t*>(h + 1024);                // kMaxTopK
  uint32_t* pre = reinterpret_cast<uint32_t*>(sel + kMaxTopK);        // kMaxChunks
  uint32_t* cbase = pre + kMaxChunks;                                 // kMaxChunks
  __shared__ uint32_t s_warp[NT / 32];
  pdl_trigger();
  pdl_wait();
  const int b = blockIdx.x, tid = threadIdx.x;
  int32_t* out = idx_out + (int64_t)b * k;
  const int64_t nb = row_len(n, b, len_div, n_max);
  const float* s = scores + (int64_t)b * stride;
  const int32_t* cp = cand_pos ? cand_pos + (int64_t)b * stride : nullptr;
  // the row header in one 16-byte load: {cnt, overflow, done, vbin}
  const uint4 hv = *reinterpret_cast<const uint4*>(hdr + b);
  // direct mode: the first eight entries of this thread, loaded before the
  // header is looked at (harmless reads of the row on the other paths)
  float v[8];
  int32_t p[8];
  if (mode == kFinDirect) load8(s, cp, (int64_t)tid * 8, nb, v, p);
  if (hv.y) {
    // slow path: count the row's present candidates, then select over global memory
    __shared__ uint32_t s_valid;
    if (tid == 0) s_valid = 0;
    __syncthreads();
    uint32_t loc = 0;
    for (int64_t i = tid; i < nb; i += NT) loc += (cp == nullptr || cp[i] >= 0);
    atomicAdd(&s_valid, loc);
    __syncthreads();
    RowKeys src{s, cp, nb};
    select_and_write<NT>(src, k, (int64_t)s_valid, out, h, sel);
    return;
  }
  const int vbin = (int)hv.w;
  int cnt = 0;
  if (mode == kFinDirect) {
    // the row itself, in index order: entries at or above the threshold bin;
    // the next 8192 entries load while these are compacted
    uint32_t run = 0;
    for (int64_t i0 = 0; i0 < nb; i0 += (int64_t)NT * 8) {
      float vn[8];
      int32_t pn[8];
      const int64_t nxt = i0 + (int64_t)NT * 8;
      if (nxt < nb) load8(s, cp, nxt + (int64_t)tid * 8, nb, vn, pn);
      uint32_t take = 0;
#pragma unroll
      for (int u = 0; u < 8; ++u)
        if (p[u] >= 0 && (int)(score_key(v[u]) >> 20) >= vbin) take |= 1u << u;
      uint32_t tot;
      uint32_t slot = run + block_excl_scan<NT>(__popc(take), s_warp, &tot);
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        if (!((take >> u) & 1)) continue;
        if (slot < (uint32_t)kCandCap) keys[slot] = cand_key(v[u], p[u]);
        ++slot;
      }
      run += tot;
      if (nxt < nb) {
#pragma unroll
        for (int u = 0; u < 8; ++u) { v[u] = vn[u]; p[u] = pn[u]; }
      }
    }
    cnt = (int)min(run, (uint32_t)kCandCap);
  } else if (mode == kFinTable) {
    // chunk order is index order: prefix of the chunk counts, then one
    // binary search per candidate into the prefix
    const int nch = (int)((nb + kChunk - 1) / kChunk);
    constexpr int kPer = kMaxChunks / NT;
    uint2 e[kPer];
    uint32_t sum = 0;
#pragma unroll
    for (int u = 0; u < kPer; ++u) {
      const int c = tid * kPer + u;
      e[u] = c < nch ? tab[(int64_t)b * kMaxChunks + c] : make_uint2(0u, 0u);
      sum += e[u].y;
    }
    uint32_t tot;
    uint32_t run = block_excl_scan<NT>(sum, s_warp, &tot);
#pragma unroll
    for (int u = 0; u < kPer; ++u) {
      const int c = tid * kPer + u;
      if (c < nch) { pre[c] = run; cbase[c] = e[u].x; }
      run += e[u].y;
    }
    __syncthreads();
    cnt = (int)min(tot, (uint32_t)kCandCap);
    const uint64_t* rc = cand + (int64_t)b * kCandCap;
    constexpr int kG = kCandCap / NT;
    uint64_t kv[kG];
#pragma unroll
    for (int u = 0; u < kG; ++u) {
      const int o = tid + u * NT;
      kv[u] = 0;
      if (o < cnt) {
        int lo = 0, hi = nch - 1;                     // last chunk with pre <= o
        while (lo < hi) {
          const int mid = (lo + hi + 1) >> 1;
          if (pre[mid] <= (uint32_t)o) lo = mid; else hi = mid - 1;
        }
        const uint32_t slot = cbase[lo] + ((uint32_t)o - pre[lo]);
        kv[u] = rc[slot < (uint32_t)kCandCap ? slot : 0];
      }
    }
#pragma unroll
    for (int u = 0; u < kG; ++u) {
      const int o = tid + u * NT;
      if (o < cnt) keys[o] = kv[u];
    }
  } else {
    cnt = (int)min(hv.x, (uint32_t)kCandCap);
    for (int i = tid; i < cnt; i += NT) keys[i] = cand[(int64_t)b * kCandCap + i];
  }
  __syncthreads();
  // positions increasing along the candidates: select in order, no sort
  bool mono = mode != kFinUnordered;
  if (mono) {
    const int S = (cnt + NT - 1) / NT;
    const int lo = min(tid * S, cnt), hi = min(lo + S + 1, cnt);
    for (int i = lo + 1; i < hi; ++i)
      if (cand_pos_of(keys[i - 1]) >= cand_pos_of(keys[i])) mono = false;
  }
  if (__syncthreads_and(mono)) {
    ordered_select<NT>(keys, cnt, vbin, k, out, h, pre, s_warp);   // the chunk prefix is no longer needed
  } else {
    SmemKeys src{keys, cnt};
    select_and_write<NT>(src, k, cnt, out, h, sel);
  }
}

int topk_final_smem() { return kCandCap * 8 + 1024 * 4 + kMaxTopK * 4 + 2 * kMaxChunks * 4; }

// ---- block scores of the max-of-token pool rule -------------------------------
// bmax[b][j] = the largest score of positions 8 j .. 8 j + 7 below n[b]: a
// block holding any of the row's Top-k positions scores at least the k-th
// score, so the best P >= k blocks hold every one of them.
__global__ void __launch_bounds__(256) k_block_max(const float* __restrict__ scores, int64_t stride,
                                                   const int64_t* __restrict__ n, int64_t n_max,
                                                   float* __restrict__ bmax, int64_t nb_max) {
  pdl_trigger();
  pdl_wait();
  const int b = blockIdx.y;
  const int64_t len = row_len(n, b, 1, n_max);
  const int64_t nblk = (len + kBlock - 1) / kBlock;
  const float* s = scores + (int64_t)b * stride;
  for (int64_t j = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; j < nblk; j += (int64_t)gridDim.x * blockDim.x) {
    const int64_t t0 = j * kBlock;
    float m = s[t0];
#pragma unroll
    for (int u = 1; u < kBlock; ++u)
      if (t0 + u < len) m = fmaxf(m, s[t0 + u]);
    bmax[(int64_t)b * nb_max + j] = m;
  }
}

// ---- host ------------------------------------------------------------------
static int64_t tk_rows_per_cta(int B, int64_t rows) {
  int64_t per = 16384;
  while (per > 1024 && (int64_t)B * ((rows + per - 1) / per) < 4 * kSMs) per /= 2;
  return per;
}

// Zero the histogram and headers of B rows (before the scan or step 1).
int topk_prepare(void* ws, int B, cudaStream_t s) {
  const size_t bytes = align256((size_t)B * kHistBins * 4) + align256((size_t)B * sizeof(TopkHdr));
  if (cudaMemsetAsync(ws, 0, bytes, s) != cudaSuccess) return CSA2_ERR_CUDA;
  return CSA2_OK;
}

// Steps 1 (unless the histogram is already in the workspace), 2 and 3.
int launch_topk(const float* scores, const int32_t* cand_pos, int64_t stride, const int64_t* n,
                int len_div, int B, int64_t n_max, int k, int32_t* idx_out, void* ws, bool hist_ready,
                cudaStream_t s) {
  if (B == 0) return CSA2_OK;
  TopkWs w = topk_ws(ws, B);
  int rc;
  if (!hist_ready) {
    if ((rc = topk_prepare(ws, B, s)) != CSA2_OK) return rc;
    const int64_t per = tk_rows_per_cta(B, n_max);
    dim3 grid((unsigned)((n_max + per - 1) / per > 0 ? (n_max + per - 1) / per : 1), (unsigned)B);
    const cudaError_t e = launch_pdl(k_topk_hist, grid, dim3(kTkThreads), 0, s, scores, cand_pos, stride, n, len_div,
                                     n_max, per, w.hist, w.hdr, k);
    count_launch();
    if ((rc = launch_status(e)) != CSA2_OK) return rc;
  }
  const int mode = n_max <= kDirectRows ? kFinDirect
                   : n_max <= (int64_t)kMaxChunks * kChunk ? kFinTable : kFinUnordered;
  if (mode != kFinDirect) {
    const int64_t nch = (n_max + kChunk - 1) / kChunk;
    int64_t per_row = (4 * kSMs + B - 1) / B;
    if (per_row > nch) per_row = nch;
    if (per_row < 1) per_row = 1;
    const cudaError_t e = launch_pdl(k_topk_compact, dim3((unsigned)per_row, (unsigned)B), dim3(kTkThreads), 0, s,
                                     scores, cand_pos, stride, n, len_div, n_max, w.hdr, w.cand, w.tab);
    count_launch();
    if ((rc = launch_status(e)) != CSA2_OK) return rc;
  }
  const bool small_k = k <= 512;
  const cudaError_t e = launch_pdl(small_k ? k_topk_final<kFinThreadsSmallK> : k_topk_final<kFinThreadsLargeK>,
                                   dim3((unsigned)B), dim3(small_k ? kFinThreadsSmallK : kFinThreadsLargeK),
                                   (size_t)topk_final_smem(), s,
                                   scores, cand_pos, stride, n, len_div, n_max, k,
                                   static_cast<const TopkHdr*>(w.hdr), static_cast<const uint64_t*>(w.cand),
                                   static_cast<const uint2*>(w.tab), mode, idx_out);
  count_launch();
  return launch_status(e);
}

// Pool by the max-of-token rule: block maxima of the scores, then the best
// P blocks (Top-K with its own histogram pass). ws: bmax [B][nb_max] then a
// Top-K workspace.
size_t pool_block_max_ws_bytes(int B, int64_t n_max) {
  const int64_t nb = (n_max + kBlock - 1) / kBlock;
  return align256((size_t)B * (size_t)nb * 4) + topk_ws_bytes(B);
}
int launch_pool_block_max(const float* scores, int64_t stride, const int64_t* n, int B, int64_t n_max, int P,
                          int32_t* pool_out, void* ws, cudaStream_t s) {
  if (B == 0) return CSA2_OK;
  const int64_t nb = (n_max + kBlock - 1) / kBlock;
  float* bmax = static_cast<float*>(ws);
  void* tk = static_cast<char*>(ws) + align256((size_t)B * (size_t)nb * 4);
  int64_t gx = (nb + 255) / 256;
  const int64_t cap = (4 * kSMs + B - 1) / B;
  if (gx > cap) gx = cap;
  if (gx < 1) gx = 1;
  const cudaError_t e = launch_pdl(k_block_max, dim3((unsigned)gx, (unsigned)B), dim3(256), 0, s, scores, stride,
                                   n, n_max, bmax, nb);
  count_launch();
  int rc = launch_status(e);
  if (rc != CSA2_OK) return rc;
  return launch_topk(bmax, nullptr, nb, n, kBlock, B, nb, P, pool_out, tk, false, s);
}

int topk_init_attributes() {
  for (auto kern : {k_topk_final<kFinThreadsSmallK>, k_topk_final<kFinThreadsLargeK>})
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, topk_final_smem()) != cudaSuccess)
      return CSA2_ERR_CUDA;
  return CSA2_OK;
}

}  // namespace csa2
