// decode_sm103.cuh -- bf16 single-token GQA decode over a per-sequence KV
// cache (split-KV), plus the log-sum-exp combine of the split partials.
//
// Method (sources cited by page title and section):
//  * GQA paper summary (azimuth.plus/paper/gqa), "Problem" and "Bottleneck":
//    each generation step must read every cached key and value, so the step
//    is bound by memory bandwidth; GQA shrinks what is read by Hq/Hkv because
//    the G query heads of a group share one K/V head.  Each CTA here streams
//    one K/V head's cached rows once and scores them against all G query
//    heads of the group.
//  * "3个GQA核心优化技巧" (blog.gitcode.com), "阶段二": num_splits splits the
//    key range so that several CTAs work on one sequence; "FlashAttention
//    Serisi" (webturing.pages.dev), "Ana fikir": each split keeps a running
//    max / sum, and partial results merge exactly through their log-sum-exp.
//
// Split kernel: one CTA per (split, kvh, b), 4 warps.  Every warp walks
// 16-key blocks of the split (block w, w+4, ...).  K and V rows are read
// straight from global memory with 16-byte vector loads (one 16 B chunk = 8
// consecutive head-dim values of one cached token); no shared-memory staging
// is needed because the loads are placed directly in mma.sync fragment
// order:
//   S^T (16 keys x 8 heads) = K (16 x D) . Q^T (D x 8)   m16n8k16, K as A
//   O^T (D x 8 heads)      += V^T (D x 16) . P^T (16 x 8) m16n8k16, V^T as A
// The head-dimension index is permuted consistently between the K fragment
// and the Q fragment (a dot product does not depend on the order of its
// terms), and between the V fragment and the output rows.  P^T is formed
// from the S^T accumulator with movmatrix (an 8x8 transpose in registers).
// The work per byte is 8 flop/B, which would need ~52 TFLOP/s of fp32 FMA
// at full HBM bandwidth, hence the tensor cores.
#pragma once

#include "common.cuh"

namespace gqa {
namespace decode {

constexpr int kWarps = 4;
constexpr int kThreads = kWarps * 32;
constexpr int kBlockKeys = 16;

struct Params {
  const __nv_bfloat16* q;       // [B, Hq, D]
  const __nv_bfloat16* kc;      // [B, Smax, Hkv, D]
  const __nv_bfloat16* vc;      // [B, Smax, Hkv, D]
  const int* seqlens;           // [B]
  __nv_bfloat16* out;           // [B, Hq, D]      (written when nsplit == 1)
  float* part_o;                // [B, Hq, nsplit, D] (written when nsplit > 1)
  float* part_lse;              // [B, Hq, nsplit]
  int B, Hq, Hkv, G, Smax;
  int nsplit, split_len;
  float scale_log2;
};

DEVI uint4 ldg_stream(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

DEVI void mma_bf16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                         uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

DEVI uint32_t movmatrix_trans(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}

DEVI uint32_t word(const uint4& v, int i) {
  return i == 0 ? v.x : (i == 1 ? v.y : (i == 2 ? v.z : v.w));
}

template <int D>
struct BlockRegs {
  uint4 k[2][D / 32];   // K rows (r, r+8), chunks c + 4q
  uint4 v[4][D / 64];   // V rows (2c, 2c+1, 2c+8, 2c+9), chunk 8*grp + r
};

// Loads one 16-key block starting at key `k0`; keys >= kend read as zero.
template <int D>
DEVI void load_block(BlockRegs<D>& R, const __nv_bfloat16* kbase, const __nv_bfloat16* vbase,
                     size_t row_stride, int k0, int kend, int r, int c) {
  const uint4 z = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int key = k0 + r + 8 * h;
    const __nv_bfloat16* row = kbase + size_t(key) * row_stride;
#pragma unroll
    for (int q = 0; q < D / 32; ++q)
      R.k[h][q] = (key < kend) ? ldg_stream(row + 8 * (c + 4 * q)) : z;
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int key = k0 + 2 * c + (i & 1) + 8 * (i >> 1);
    const __nv_bfloat16* row = vbase + size_t(key) * row_stride;
#pragma unroll
    for (int grp = 0; grp < D / 64; ++grp)
      R.v[i][grp] = (key < kend) ? ldg_stream(row + 8 * (8 * grp + r)) : z;
  }
}

template <int D>
__global__ void __launch_bounds__(kThreads)
    decode_split_kernel(const Params p) {
  constexpr int KS = D / 16;      // k-steps of the QK^T product
  constexpr int MT = D / 16;      // m-tiles of O^T
  const int split = blockIdx.x;
  const int kvh = blockIdx.y;
  const int b = blockIdx.z;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int r = lane >> 2;
  const int c = lane & 3;

  int Lb = p.seqlens[b];
  if (Lb < 0 || Lb > p.Smax) {
    if (split == 0 && kvh == 0 && threadIdx.x == 0) raise_error(kErrBounds);
    Lb = 0;
  }
  const int kstart = split * p.split_len;
  if (kstart >= Lb && p.nsplit > 1) return;  // empty split: the combine skips it
  const int kend = min(Lb, kstart + p.split_len);
  const int nblk = kend > kstart ? (kend - kstart + kBlockKeys - 1) / kBlockKeys : 0;

  // Q^T fragments for the G heads of this group (head n = r; zero if n >= G)
  uint32_t qf[KS][2];
  {
    const bool hv = r < p.G;
    const __nv_bfloat16* qrow = p.q + (size_t(b) * p.Hq + size_t(kvh) * p.G + (hv ? r : 0)) * D;
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
      const int d0 = 8 * (c + 4 * (ks >> 1)) + 4 * (ks & 1);
      uint2 w = hv ? *reinterpret_cast<const uint2*>(qrow + d0) : make_uint2(0u, 0u);
      qf[ks][0] = w.x;
      qf[ks][1] = w.y;
    }
  }

  const size_t row_stride = size_t(p.Hkv) * D;
  const __nv_bfloat16* kbase = p.kc + (size_t(b) * p.Smax * p.Hkv + kvh) * D;
  const __nv_bfloat16* vbase = p.vc + (size_t(b) * p.Smax * p.Hkv + kvh) * D;
  const float cl = p.scale_log2;

  float o[MT][4];
#pragma unroll
  for (int mt = 0; mt < MT; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;
  float mA = -INFINITY, mB = -INFINITY, lA = 0.f, lB = 0.f;   // heads 2c and 2c+1

  BlockRegs<D> cur, nxt;
  int blk = warp;
  if (blk < nblk) load_block<D>(cur, kbase, vbase, row_stride, kstart + blk * kBlockKeys, kend, r, c);
  for (; blk < nblk; blk += kWarps) {
    const int nb = blk + kWarps;
    if (nb < nblk) load_block<D>(nxt, kbase, vbase, row_stride, kstart + nb * kBlockKeys, kend, r, c);
    const int k0 = kstart + blk * kBlockKeys;

    // S^T = K . Q^T
    float s[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
      const int q = ks >> 1, hw = 2 * (ks & 1);
      mma_bf16_16816(s, word(cur.k[0][q], hw), word(cur.k[1][q], hw), word(cur.k[0][q], hw + 1),
                     word(cur.k[1][q], hw + 1), qf[ks][0], qf[ks][1]);
    }
    // scale, mask, online softmax per head (max over the 16 keys of the block)
    const bool v0 = (k0 + r) < kend, v1 = (k0 + r + 8) < kend;
    const float tA0 = v0 ? s[0] * cl : -INFINITY, tB0 = v0 ? s[1] * cl : -INFINITY;
    const float tA1 = v1 ? s[2] * cl : -INFINITY, tB1 = v1 ? s[3] * cl : -INFINITY;
    float xA = fmaxf(tA0, tA1), xB = fmaxf(tB0, tB1);
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
      xA = fmaxf(xA, __shfl_xor_sync(0xffffffffu, xA, off));
      xB = fmaxf(xB, __shfl_xor_sync(0xffffffffu, xB, off));
    }
    const float nA = fmaxf(mA, xA), nB = fmaxf(mB, xB);
    const float rA = (nA == -INFINITY) ? 0.f : nA, rB = (nB == -INFINITY) ? 0.f : nB;
    const float aA = ex2_approx(mA - rA), aB = ex2_approx(mB - rB);
    mA = nA;
    mB = nB;
    const float pA0 = ex2_approx(tA0 - rA), pA1 = ex2_approx(tA1 - rA);
    const float pB0 = ex2_approx(tB0 - rB), pB1 = ex2_approx(tB1 - rB);
    lA = lA * aA + pA0 + pA1;
    lB = lB * aB + pB0 + pB1;
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) {
      o[mt][0] *= aA;
      o[mt][1] *= aB;
      o[mt][2] *= aA;
      o[mt][3] *= aB;
    }
    // P^T fragments: transpose the two 8x8 (key x head) halves of P
    const uint32_t pb0 = movmatrix_trans(pack_bf16x2(pA0, pB0));
    const uint32_t pb1 = movmatrix_trans(pack_bf16x2(pA1, pB1));
    // O^T += V^T . P^T
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) {
      const int grp = mt >> 2, tt = mt & 3;
      const uint32_t w0 = word(cur.v[0][grp], tt), w1 = word(cur.v[1][grp], tt);
      const uint32_t w2 = word(cur.v[2][grp], tt), w3 = word(cur.v[3][grp], tt);
      mma_bf16_16816(o[mt], __byte_perm(w0, w1, 0x5410), __byte_perm(w0, w1, 0x7632),
                     __byte_perm(w2, w3, 0x5410), __byte_perm(w2, w3, 0x7632), pb0, pb1);
    }
    if (nb < nblk) cur = nxt;
  }

  // per-warp totals of l over the 8 lanes that share c
#pragma unroll
  for (int off = 4; off < 32; off <<= 1) {
    lA += __shfl_xor_sync(0xffffffffu, lA, off);
    lB += __shfl_xor_sync(0xffffffffu, lB, off);
  }

  // ---- combine the 4 warps through shared memory
  __shared__ float s_o[kWarps][8][D];
  __shared__ float s_m[kWarps][8];
  __shared__ float s_l[kWarps][8];
#pragma unroll
  for (int mt = 0; mt < MT; ++mt) {
    const int grp = mt >> 2, tt = mt & 3;
    const int d_lo = 64 * grp + 8 * r + 2 * tt;   // row m = r ; row m = r + 8 is d_lo + 1
    s_o[warp][2 * c][d_lo] = o[mt][0];
    s_o[warp][2 * c + 1][d_lo] = o[mt][1];
    s_o[warp][2 * c][d_lo + 1] = o[mt][2];
    s_o[warp][2 * c + 1][d_lo + 1] = o[mt][3];
  }
  if (r == 0) {
    s_m[warp][2 * c] = mA;
    s_m[warp][2 * c + 1] = mB;
    s_l[warp][2 * c] = lA;
    s_l[warp][2 * c + 1] = lB;
  }
  __syncthreads();

  const int G = p.G;
  for (int idx = threadIdx.x; idx < G * D; idx += kThreads) {
    const int n = idx / D, d = idx % D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) M = fmaxf(M, s_m[w][n]);
    const float Mr = (M == -INFINITY) ? 0.f : M;
    float num = 0.f, den = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      const float f = ex2_approx(s_m[w][n] - Mr);
      num += f * s_o[w][n][d];
      den += f * s_l[w][n];
    }
    const float val = den > 0.f ? num / den : 0.f;
    const size_t hrow = size_t(b) * p.Hq + size_t(kvh) * G + n;
    if (p.nsplit == 1) {
      p.out[hrow * D + d] = __float2bfloat16_rn(val);
    } else {
      p.part_o[(hrow * p.nsplit + split) * D + d] = val;
      if (d == 0)
        p.part_lse[hrow * p.nsplit + split] =
            den > 0.f ? (Mr + log2f(den)) * 0.6931471805599453f : -INFINITY;
    }
  }
}

// Log-sum-exp combine of split partials: one warp per (b, h).
//   lse = ln sum_s exp(lse_s);  out = sum_s exp(lse_s - lse) * O_s
// Splits whose start is at or past the sequence length were never written
// and are skipped.  OutT is __nv_bfloat16 or float.
template <typename OutT>
__global__ void __launch_bounds__(128)
    combine_kernel(const float* part_o, const float* part_lse, const int* seqlens, OutT* out,
                   int B, int Hq, int D, int nsplit, int split_len, int Smax) {
  const int row = blockIdx.x * 4 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= B * Hq) return;
  const int b = row / Hq;
  int Lb = seqlens[b];
  if (Lb < 0 || Lb > Smax) Lb = 0;
  const int nvalid = min(nsplit, (Lb + split_len - 1) / split_len);
  const float* lrow = part_lse + size_t(row) * nsplit;
  float M = -INFINITY;
  for (int s = 0; s < nvalid; ++s) M = fmaxf(M, lrow[s]);
  float W = 0.f;
  const float Mr = (M == -INFINITY) ? 0.f : M;
  for (int s = 0; s < nvalid; ++s) W += expf(lrow[s] - Mr);
  const float inv = W > 0.f ? 1.f / W : 0.f;
  for (int d = lane; d < D; d += 32) {
    float acc = 0.f;
    for (int s = 0; s < nvalid; ++s)
      acc += expf(lrow[s] - Mr) * part_o[(size_t(row) * nsplit + s) * D + d];
    const float val = acc * inv;
    if constexpr (sizeof(OutT) == 2)
      out[size_t(row) * D + d] = __float2bfloat16_rn(val);
    else
      out[size_t(row) * D + d] = val;
  }
}

}  // namespace decode
}  // namespace gqa
