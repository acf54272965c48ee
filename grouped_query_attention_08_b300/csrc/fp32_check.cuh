// fp32_check.cuh -- exact-fp32 SIMT grouped-query attention (prefill and
// decode), the library's float32 check mode.
//
// Same method as the bf16 kernels -- K/V head kvh = h / G ("3个GQA核心优化技巧",
// blog.gitcode.com, "Flash-Attention的稀疏分组优化"), scores scale * q.k,
// masked keys excluded, an online (running max / running sum) softmax over
// the keys ("FlashAttention Serisi", webturing.pages.dev, "Ana fikir") -- in
// plain fp32 on the CUDA cores, with no rounding of P or of the inputs.
//
// One warp per (b, h, i) row and key split; the lanes split the head
// dimension (d = lane + 32 e) and each score is a warp-wide sum.
#pragma once

#include "common.cuh"

namespace gqa {
namespace f32 {

constexpr int kWarps = 8;
constexpr int kMaxD = 256;

struct Params {
  const float* q;
  const float* k;
  const float* v;
  float* out;          // final output (nsplit == 1), same layout as q
  float* lse;          // [B, Hq, Sq] or nullptr (nsplit == 1)
  float* part_o;       // [B*Hq*Sq rows, nsplit, D] (nsplit > 1)
  float* part_lse;     // [rows, nsplit]
  const int* seqlens;  // [B] or nullptr
  long long q_sb, q_ss, q_sh;   // element strides of q/out: batch, token, head
  long long k_sb, k_ss, k_sh;   // element strides of k/v: batch, key, kv head
  int B, Hq, Hkv, G, Sq, Sk, D, causal;
  float scale;
  int nsplit, split_len;
  int len_cap;         // largest legal key length (Sk, or the cache capacity)
};

__global__ void __launch_bounds__(kWarps * 32) attention_kernel(const Params p) {
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const long long row = (long long)blockIdx.x * kWarps + warp;   // (b * Hq + h) * Sq + i
  const long long nrows = (long long)p.B * p.Hq * p.Sq;
  if (row >= nrows) return;
  const int split = blockIdx.y;
  const int i = int(row % p.Sq);
  const int h = int((row / p.Sq) % p.Hq);
  const int b = int(row / ((long long)p.Sq * p.Hq));
  const int kvh = h / p.G;

  int Lb = p.seqlens ? p.seqlens[b] : p.Sk;
  if (Lb < 0 || Lb > p.len_cap) {
    if (lane == 0 && i == 0 && h == 0 && split == 0) raise_error(kErrBounds);
    Lb = 0;
  }
  int lim = Lb;
  if (p.causal) lim = min(lim, i + p.Sk - p.Sq + 1);
  lim = max(lim, 0);
  const int j0 = split * p.split_len;
  const int j1 = min(lim, j0 + p.split_len);

  constexpr int E = kMaxD / 32;
  float qv[E], ov[E];
  const float* qrow = p.q + b * p.q_sb + (long long)i * p.q_ss + (long long)h * p.q_sh;
#pragma unroll
  for (int e = 0; e < E; ++e) {
    const int d = lane + 32 * e;
    qv[e] = d < p.D ? qrow[d] : 0.f;
    ov[e] = 0.f;
  }
  const float* kb = p.k + b * p.k_sb + (long long)kvh * p.k_sh;
  const float* vb = p.v + b * p.k_sb + (long long)kvh * p.k_sh;
  float m = -INFINITY, l = 0.f;
  for (int j = j0; j < j1; ++j) {
    const float* kr = kb + (long long)j * p.k_ss;
    float part = 0.f;
#pragma unroll
    for (int e = 0; e < E; ++e) {
      const int d = lane + 32 * e;
      if (d < p.D) part = fmaf(qv[e], kr[d], part);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) part += __shfl_xor_sync(0xffffffffu, part, off);
    const float s = part * p.scale;
    const float mn = fmaxf(m, s);
    const float alpha = expf(m - mn);     // m = -inf on the first key: alpha = 0
    const float pj = expf(s - mn);
    l = l * alpha + pj;
    const float* vr = vb + (long long)j * p.k_ss;
#pragma unroll
    for (int e = 0; e < E; ++e) {
      const int d = lane + 32 * e;
      if (d < p.D) ov[e] = fmaf(pj, vr[d], ov[e] * alpha);
    }
    m = mn;
  }
  const float inv = l > 0.f ? 1.f / l : 0.f;
  const float lse = l > 0.f ? m + logf(l) : -INFINITY;
  if (p.nsplit == 1) {
    float* orow = p.out + b * p.q_sb + (long long)i * p.q_ss + (long long)h * p.q_sh;
#pragma unroll
    for (int e = 0; e < E; ++e) {
      const int d = lane + 32 * e;
      if (d < p.D) orow[d] = ov[e] * inv;
    }
    if (p.lse && lane == 0) p.lse[row] = lse;
  } else {
    float* prow = p.part_o + (row * p.nsplit + split) * p.D;
#pragma unroll
    for (int e = 0; e < E; ++e) {
      const int d = lane + 32 * e;
      if (d < p.D) prow[d] = ov[e] * inv;
    }
    if (lane == 0) p.part_lse[row * p.nsplit + split] = lse;
  }
}

}  // namespace f32
}  // namespace gqa
