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
// [b][split][dim / 4][H][4] and (m, l) as [b][split][H][2]; one thread per
// (four dims, head) with heads fastest, so a warp's loads are contiguous. The
// kernel is bound by load latency: U splits' loads are all issued before any
// is used (U >= splits for decode shapes: one round trip), with an online
// rescale across rounds when there are more splits than U.
template <int U>
__global__ void __launch_bounds__(128) k_attn_merge(const float* __restrict__ part_o,
                                                    const float* __restrict__ part_ml, int H, int splits,
                                                    __nv_bfloat16* __restrict__ out) {
  pdl_trigger();
  pdl_wait();
  const int b = blockIdx.y;
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= (kD / 4) * H) return;
  const int d4 = i / H, h = i - d4 * H;
  const float* ml = part_ml + ((int64_t)b * splits * H + h) * 2;
  const float* po = part_o + ((int64_t)b * splits * (kD / 4) + d4) * H * 4 + h * 4;
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
int launch_sparse_attn_tc(const void* q, int B, int H, const uint8_t* codes, const uint8_t* scales,
                          int64_t kv_seq_stride, int64_t n_cap, const int32_t* idx, int k, const void* swa,
                          int64_t swa_seq_stride, int W, int swa_tail, int rps, const int32_t* swa_len,
                          float softmax_scale, void* out, float* part_o, float* part_ml, int splits, int tps,
                          int32_t* st, cudaStream_t s);

// Split-K count. The attention kernel runs one CTA per SM (its shared memory
// and all 512 TMEM columns). A batch that fills the machine runs unsplit (a
// split writes an fp32 partial of H x 512 per CTA and needs the merge pass).
// Otherwise minimise waves x tiles per split plus one tile-equivalent for
// the merge; ties go to fewer splits.
int attn_splits(int B, int H, int k, int W) {
  (void)H;
  const int n_tiles = (k + W + kTile - 1) / kTile;
  const int64_t slots = kSMs;
  if ((int64_t)B >= slots) return 1;
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

size_t attn_ws_bytes(int B, int H, int k, int W) {
  const int s = attn_splits(B, H, k, W);
  if (s <= 1) return 0;
  const size_t po = (size_t)B * s * H * kD * 4;
  return ((po + 255) & ~(size_t)255) + (size_t)B * s * H * 2 * 4;
}

int launch_sparse_attn(const void* q, int B, int H, const uint8_t* codes, const uint8_t* scales,
                       int64_t kv_seq_stride, int64_t n_cap, const int32_t* idx, int k, const void* swa,
                       int64_t swa_seq_stride, int W, int swa_tail, int rps, const int32_t* swa_len,
                       float softmax_scale, void* out, void* ws, int32_t* st, cudaStream_t s) {
  if (B == 0) return CSA2_OK;
  if (H < 1 || H > 64) return CSA2_ERR_UNSUPPORTED_SHAPE;
  const int splits = attn_splits(B, H, k, W);
  const int n_tiles = (k + W + kTile - 1) / kTile;
  const int tps = (n_tiles + splits - 1) / splits;
  float* part_o = nullptr;
  float* part_ml = nullptr;
  if (splits > 1) {
    part_o = static_cast<float*>(ws);
    const size_t po = (size_t)B * splits * H * kD * 4;
    part_ml = reinterpret_cast<float*>(static_cast<char*>(ws) + ((po + 255) & ~(size_t)255));
  }
  int rc = launch_sparse_attn_tc(q, B, H, codes, scales, kv_seq_stride, n_cap, idx, k, swa, swa_seq_stride, W,
                                 swa_tail, rps < 1 ? 1 : rps, swa_len, softmax_scale, out, part_o, part_ml, splits,
                                 tps, st, s);
  if (rc != CSA2_OK || splits == 1) return rc;
  const dim3 grid((unsigned)(((kD / 4) * H + 127) / 128), (unsigned)B);
  auto kern = splits <= 4 ? k_attn_merge<4> : splits <= 8 ? k_attn_merge<8> : k_attn_merge<16>;
  const cudaError_t e = launch_pdl(kern, grid, dim3(128), 0, s, static_cast<const float*>(part_o),
                                   static_cast<const float*>(part_ml), H, splits,
                                   reinterpret_cast<__nv_bfloat16*>(out));
  count_launch();
  return launch_status(e);
}

}  // namespace csa2
