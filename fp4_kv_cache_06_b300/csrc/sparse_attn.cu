// sparse_attn.cu — host dispatch of the CSA2 sparse attention (the kernel is
// k_sparse_attn_tc in sparse_attn_tc.cu) and the log-sum-exp merge of its
// split-K partials.
//
// [CSA2] wire.sakhanda.co, "DeepSeek AI выпустила DeepSeek-V4.1-Flash ...",
//        section "Сжатое разреженное внимание 2 (CSA2)": each layer attends
//        over the Top-512 main-KV entries plus its own SWA KV. Splitting the
//        key slots across CTAs and merging the partial (m, l, O) by
//        log-sum-exp is exact.
#include "common.cuh"

namespace csa2 {

constexpr int kD = 512;          // main head dim
constexpr int kTile = 64;        // keys per tile of the attention kernel

// Log-sum-exp merge of split-K partials. Partial O is stored
// [layer][b][split][dim / 4][H][4] and (m, l) as [layer][b][split][H][2]
// (layer = blockIdx.z, b = blockIdx.y); one thread per
// (four dims, head) with heads fastest, so a warp's loads are contiguous. The
// kernel is bound by load latency: U splits' loads are all issued before any
// is used (U >= splits for decode shapes: one round trip), with an online
// rescale across rounds when there are more splits than U.
template <int U>
__global__ void __launch_bounds__(128) k_attn_merge(const float* __restrict__ part_o,
                                                    const float* __restrict__ part_ml, int H, int splits,
                                                    const AttnLayers lay) {
  pdl_trigger();
  pdl_wait();
  const int b = blockIdx.y;
  const int64_t unit = (int64_t)blockIdx.z * gridDim.y + b;
  __nv_bfloat16* __restrict__ out = lay.out[blockIdx.z];
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= (kD / 4) * H) return;
  const int d4 = i / H, h = i - d4 * H;
  const float* ml = part_ml + (unit * splits * H + h) * 2;
  const float* po = part_o + (unit * splits * (kD / 4) + d4) * H * 4 + h * 4;
  const int64_t po_split = (int64_t)(kD / 4) * H * 4;
  float M = -INFINITY, Lsum = 0.f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int s0 = 0; s0 < splits; s0 += U) {
    float m[U], l[U];
    float4 v[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      m[u] = -INFINITY;
      l[u] = 0.f;
      v[u] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (s0 + u < splits) {
        const float2 x = *reinterpret_cast<const float2*>(ml + (int64_t)(s0 + u) * H * 2);
        m[u] = x.x;
        l[u] = x.y;
        v[u] = *reinterpret_cast<const float4*>(po + (s0 + u) * po_split);
      }
    }
    float Mc = M;
#pragma unroll
    for (int u = 0; u < U; ++u) Mc = fmaxf(Mc, m[u]);
    if (Mc == -INFINITY) continue;                   // nothing attended so far
    const float sc = exp2f(M - Mc);                  // 0 while M is still -inf
    Lsum *= sc;
    acc.x *= sc; acc.y *= sc; acc.z *= sc; acc.w *= sc;
#pragma unroll
    for (int u = 0; u < U; ++u) {
      if (m[u] == -INFINITY) continue;
      const float wgt = exp2f(m[u] - Mc);
      Lsum += wgt * l[u];
      acc.x += wgt * v[u].x; acc.y += wgt * v[u].y; acc.z += wgt * v[u].z; acc.w += wgt * v[u].w;
    }
    M = Mc;
  }
  const float inv = Lsum > 0.f ? 1.f / Lsum : 0.f;
  __nv_bfloat16* o = out + ((int64_t)b * H + h) * kD + 4 * d4;
  *reinterpret_cast<__nv_bfloat162*>(o) = __floats2bfloat162_rn(acc.x * inv, acc.y * inv);
  *reinterpret_cast<__nv_bfloat162*>(o + 2) = __floats2bfloat162_rn(acc.z * inv, acc.w * inv);
}

// ---- host ------------------------------------------------------------------
int launch_sparse_attn_tc(const AttnLayers& lay, int L, int B, int H, const uint8_t* codes, const uint8_t* scales,
                          int64_t kv_seq_stride, int64_t n_cap, const int32_t* idx, int k, int64_t swa_seq_stride,
                          int W, int swa_tail, int rps, const int32_t* swa_len, float softmax_scale, float* part_o,
                          float* part_ml, int splits, int tps, int32_t* st, uint64_t wait_ns, int fault,
                          int early, cudaStream_t s);

// Split-K count for `units` = rows x layers of one launch. The attention
// kernel runs one CTA per SM (its shared memory and all 512 TMEM columns). A
// launch that fills the machine runs unsplit (a split writes an fp32 partial
// of H x 512 per CTA and needs the merge pass). Otherwise minimise
// waves x tiles per split plus one tile-equivalent for the merge; ties go to
// fewer splits.
int attn_splits(int64_t units, int H, int k, int W) {
  (void)H;
  const int n_tiles = (k + W + kTile - 1) / kTile;
  const int64_t slots = kSMs;
  if (units >= slots) return 1;
  const int64_t B = units;
  int best = 1;
  int64_t best_cost = -1;
  for (int s = 1; s <= n_tiles; ++s) {
    const int tps = (n_tiles + s - 1) / s;
    const int sp = (n_tiles + tps - 1) / tps;  // splits actually holding tiles
    if (sp != s) continue;
    const int64_t waves = ((int64_t)B * s + slots - 1) / slots;
    const int64_t cost = waves * tps + (s > 1 ? 1 : 0);
    if (best_cost < 0 || cost < best_cost) { best_cost = cost; best = s; }
  }
  return best;
}

// Partials of one launch over `units` = rows x layers.
size_t attn_ws_bytes(int64_t units, int H, int k, int W) {
  const int s = attn_splits(units, H, k, W);
  if (s <= 1) return 0;
  const size_t po = (size_t)units * s * H * kD * 4;
  return ((po + 255) & ~(size_t)255) + (size_t)units * s * H * 2 * 4;
}

// Partials of a group of any size over B rows: the group is attended
// kMaxAttnLayers layers per launch, so the largest launch has at most that many.
size_t attn_group_ws_bytes(int64_t B, int H, int k, int W) {
  size_t m = 0;
  for (int L = 1; L <= kMaxAttnLayers; ++L) {
    const size_t a = attn_ws_bytes(B * L, H, k, W);
    if (a > m) m = a;
  }
  return m;
}

// Layers 0 .. L - 1 of `lay` (L <= kMaxAttnLayers) over rows 0 .. B - 1.
// `early`: the kernels of the same call that precede this launch write only
// `idx` (and the workspace), and the call's first kernel is an ordinary
// launch, which begins after all earlier work on the stream: then every
// other input was complete before the attention kernel can start, and it
// reads them before waiting for its predecessor.
int launch_sparse_attn(const AttnLayers& lay, int L, int B, int H, const uint8_t* codes, const uint8_t* scales,
                       int64_t kv_seq_stride, int64_t n_cap, const int32_t* idx, int k, int64_t swa_seq_stride,
                       int W, int swa_tail, int rps, const int32_t* swa_len, float softmax_scale, void* ws,
                       int32_t* st, bool early, cudaStream_t s) {
  if (B == 0 || L == 0) return CSA2_OK;
  if (H < 1 || H > 64 || L < 0 || L > kMaxAttnLayers || B > 65535) return CSA2_ERR_UNSUPPORTED_SHAPE;
  const int64_t units = (int64_t)B * L;
  const int splits = attn_splits(units, H, k, W);
  const int n_tiles = (k + W + kTile - 1) / kTile;
  const int tps = (n_tiles + splits - 1) / splits;
  float* part_o = nullptr;
  float* part_ml = nullptr;
  if (splits > 1) {
    part_o = static_cast<float*>(ws);
    const size_t po = (size_t)units * splits * H * kD * 4;
    part_ml = reinterpret_cast<float*>(static_cast<char*>(ws) + ((po + 255) & ~(size_t)255));
  }
  int rc = launch_sparse_attn_tc(lay, L, B, H, codes, scales, kv_seq_stride, n_cap, idx, k, swa_seq_stride, W,
                                 swa_tail, rps < 1 ? 1 : rps, swa_len, softmax_scale, part_o, part_ml, splits, tps,
                                 st, debug_wait_ns(), debug_fault() == kFaultAttn ? 1 : 0, early ? 1 : 0, s);
  if (rc != CSA2_OK || splits == 1) return rc;
  const dim3 grid((unsigned)(((kD / 4) * H + 127) / 128), (unsigned)B, (unsigned)L);
  auto kern = splits <= 4 ? k_attn_merge<4> : splits <= 8 ? k_attn_merge<8> : k_attn_merge<16>;
  const cudaError_t e = launch_pdl(kern, grid, dim3(128), 0, s, static_cast<const float*>(part_o),
                                   static_cast<const float*>(part_ml), H, splits, lay);
  count_launch();
  return launch_status(e);
}

}  // namespace csa2
