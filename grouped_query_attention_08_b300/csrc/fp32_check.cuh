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
  const int* seqlens;  // [B] or nullptr (dense layout)
  // Packed layout when cu_q != nullptr: q/out [total_q, Hq, D], k/v
  // [total_k, Hkv, D], lse [Hq, total_q]; sequence b owns query rows
  // [cu_q[b], cu_q[b+1]) and key rows [cu_k[b], cu_k[b+1]); Sq / Sk are the
  // largest sequence lengths.
  const int* cu_q;
  const int* cu_k;
  int total_q, total_k;
  // block sparsity (dense layout): key j is a candidate for query i only
  // when bmask[(i / bs) * n_kb + j / bs] != 0
  const uint8_t* bmask;
  int bs, n_kb;
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
  // dense: row = (b * Hq + h) * Sq + i;  packed: row = h * total_q + packed row
  const long long row = (long long)blockIdx.x * kWarps + warp;
  const long long nrows = p.cu_q ? (long long)p.Hq * p.total_q : (long long)p.B * p.Hq * p.Sq;
  if (row >= nrows) return;
  const int split = blockIdx.y;
  int i, h, b, Lb, diag;
  long long q_off, k_off;       // element offsets of the row's query and of the sequence's key 0
  bool ok = true;
  if (p.cu_q) {
    h = int(row / p.total_q);
    const int gi = int(row % p.total_q);
    int lo = 0, hi = p.B;     // last b with cu_q[b] <= gi
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (p.cu_q[mid] <= gi) lo = mid; else hi = mid;
    }
    if (gi >= p.cu_q[p.B]) return;   // a packed row after the last sequence: not written
    b = lo;
    const int qs = p.cu_q[b], qe = p.cu_q[b + 1], ks = p.cu_k[b], ke = p.cu_k[b + 1];
    i = gi - qs;
    Lb = ke - ks;
    const int Lq = qe - qs;
    ok = qs >= 0 && qs <= gi && gi < qe && Lq <= p.Sq && ks >= 0 && Lb >= 0 && Lb <= p.len_cap && ke <= p.total_k;
    diag = Lb - Lq;
    q_off = (long long)gi * p.q_ss + (long long)h * p.q_sh;
    k_off = (long long)ks * p.k_ss;
  } else {
    i = int(row % p.Sq);
    h = int((row / p.Sq) % p.Hq);
    b = int(row / ((long long)p.Sq * p.Hq));
    Lb = p.seqlens ? p.seqlens[b] : p.Sk;
    ok = Lb >= 0 && Lb <= p.len_cap;
    diag = p.Sk - p.Sq;
    q_off = b * p.q_sb + (long long)i * p.q_ss + (long long)h * p.q_sh;
    k_off = b * p.k_sb;
  }
  const int kvh = h / p.G;
  if (!ok) {
    if (lane == 0 && split == 0 && (p.cu_q || (i == 0 && h == 0))) raise_error(kErrBounds);
    Lb = 0;
  }
  int lim = Lb;
  if (p.causal) lim = min(lim, i + diag + 1);
  lim = max(lim, 0);
  const int j0 = split * p.split_len;
  const int j1 = min(lim, j0 + p.split_len);

  constexpr int E = kMaxD / 32;
  float qv[E], ov[E];
  const float* qrow = p.q + q_off;
#pragma unroll
  for (int e = 0; e < E; ++e) {
    const int d = lane + 32 * e;
    qv[e] = d < p.D ? qrow[d] : 0.f;
    ov[e] = 0.f;
  }
  const float* kb = p.k + k_off + (long long)kvh * p.k_sh;
  const float* vb = p.v + k_off + (long long)kvh * p.k_sh;
  float m = -INFINITY, l = 0.f;
  const uint8_t* mrow = p.bmask ? p.bmask + (size_t)(i / p.bs) * p.n_kb : nullptr;
  for (int j = j0; j < j1; ++j) {
    if (mrow && !mrow[j / p.bs]) continue;
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
    float* orow = p.out + q_off;
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
