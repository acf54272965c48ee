// backward_sm103.cuh -- gradients of the GQA forward (dQ, dK, dV), bf16.
//
// Sources (page title and section): "FlashAttention Serisi"
// (webturing.pages.dev), "V2" (a faster backward pass is one of its gains)
// and "Ana fikir" (the softmax intermediates stay out of slow memory; read
// here as: the weights are rebuilt from the forward's log-sum-exp, nothing
// quadratic is stored); "3个GQA核心优化技巧"
// (blog.gitcode.com), "GQA的分组共享机制": the G query heads of a group
// share one K/V head, so that head's gradient is the sum over the group.
//
// With P_ij = exp(scale q_i.k_j - lse_i) over the admissible keys (lse from
// the forward), Dsum_i = dO_i . O_i:
//   dV_j = sum_{h in group, i} P_ij dO_i
//   dS_ij = P_ij (dO_i . v_j - Dsum_i)
//   dQ_i = scale sum_j dS_ij k_j,   dK_j = scale sum_{h in group, i} dS_ij q_i
// Three kernels, no atomics: Dsum per query row; dQ per (b, h, 64 queries)
// looping over key tiles; dK and dV per (b, kvh, 64 keys) looping over the
// group's heads and the query tiles.  Tiles are staged in shared memory and
// multiplied with WMMA (16x16x16 bf16, fp32 accumulate); P and dS are
// rounded to bf16 for the products.
#pragma once

#include <mma.h>

#include "common.cuh"

namespace gqa {
namespace bwd {

namespace wm = nvcuda::wmma;

constexpr int kT = 64;          // queries per dQ CTA, keys per dK/dV CTA, tile edge
constexpr int kWarps = 4;       // 16 rows each
constexpr int kThreads = kWarps * 32;

struct Params {
  const __nv_bfloat16* q;       // [B, Sq, Hq, D]
  const __nv_bfloat16* k;       // [B, Sk, Hkv, D]
  const __nv_bfloat16* v;       // [B, Sk, Hkv, D]
  const __nv_bfloat16* o;       // [B, Sq, Hq, D]  forward output
  const __nv_bfloat16* dout;    // [B, Sq, Hq, D]
  const float* lse;             // [B, Hq, Sq]     forward log-sum-exp (natural log)
  const int* seqlens;           // [B] or nullptr
  float* dsum;                  // [B, Hq, Sq]     workspace
  __nv_bfloat16* dq;            // [B, Sq, Hq, D]
  __nv_bfloat16* dk;            // [B, Sk, Hkv, D]
  __nv_bfloat16* dv;            // [B, Sk, Hkv, D]
  int B, Hq, Hkv, G, Sq, Sk, causal;
  float scale;
};

template <int D>
struct Smem {
  static constexpr int kLd = D + 8;          // bf16 tile row (elements); 16-row steps stay 32-byte aligned
  static constexpr int kLdS = kT + 4;        // fp32 score tile row (elements)
  static constexpr int kTile = kT * kLd;     // elements of a 64 x D bf16 tile
  // a: Q (dQ) or K (dK/dV); b: dO or V; c: K or Q; d: V or dO (bf16 tiles);
  // per warp a 16 x 64 fp32 S tile, a 16 x 64 fp32 dP tile, two 16 x 64 bf16 tiles
  static constexpr size_t kBytes = 4 * size_t(kTile) * 2 + kWarps * (2 * 16 * kLdS * 4 + 2 * 16 * (kT + 8) * 2) +
                                   2 * kT * 4;
};

DEVI int key_len(const Params& p, int b) {
  int L = p.seqlens ? p.seqlens[b] : p.Sk;
  if (L < 0 || L > p.Sk) {
    raise_error(kErrBounds);
    L = 0;
  }
  return L;
}

// Rows [r0, r0 + 64) of the [S, H, D] slice `head` of batch b into a
// padded shared-memory tile; rows >= S are zero.  16-byte loads.
template <int D>
DEVI void load_tile(__nv_bfloat16* dst, const __nv_bfloat16* src, int b, int S, int H, int head, int r0) {
  constexpr int kChunks = D / 8;
  for (int e = threadIdx.x; e < kT * kChunks; e += kThreads) {
    const int r = e / kChunks, c = e % kChunks;
    uint4 w = make_uint4(0u, 0u, 0u, 0u);
    if (r0 + r < S) w = *reinterpret_cast<const uint4*>(src + ((size_t(b) * S + r0 + r) * H + head) * D + 8 * c);
    *reinterpret_cast<uint4*>(dst + r * Smem<D>::kLd + 8 * c) = w;
  }
}

// Dsum_i = dO_i . O_i, one warp per (b, h, i).
template <int D>
__global__ void __launch_bounds__(256) dsum_kernel(const Params p) {
  const long long row = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= (long long)p.B * p.Hq * p.Sq) return;
  const int i = int(row % p.Sq);
  const int h = int((row / p.Sq) % p.Hq);
  const int b = int(row / ((long long)p.Sq * p.Hq));
  const size_t off = ((size_t(b) * p.Sq + i) * p.Hq + h) * D;
  float acc = 0.f;
  for (int d = lane; d < D; d += 32)
    acc += __bfloat162float(p.dout[off + d]) * __bfloat162float(p.o[off + d]);
#pragma unroll
  for (int s = 16; s > 0; s >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, s);
  if (lane == 0) p.dsum[row] = acc;
}

// Shared-memory carve-up: four bf16 64 x D tiles, then per warp an fp32
// S tile, an fp32 dP tile and two bf16 16 x 64 tiles, then two fp32 row
// vectors of 64 (lse and Dsum of the tile's query rows).
template <int D>
struct Carve {
  __nv_bfloat16* t[4];
  float* s;
  float* dp;
  __nv_bfloat16* x;
  __nv_bfloat16* y;
  float* lse;
  float* dsum;
  DEVI Carve(uint8_t* base, int warp) {
    using SM = Smem<D>;
    __nv_bfloat16* tb = reinterpret_cast<__nv_bfloat16*>(base);
    for (int i = 0; i < 4; ++i) t[i] = tb + i * SM::kTile;
    uint8_t* w = base + 4 * size_t(SM::kTile) * 2 +
                 size_t(warp) * (2 * 16 * SM::kLdS * 4 + 2 * 16 * (kT + 8) * 2);
    s = reinterpret_cast<float*>(w);
    dp = s + 16 * SM::kLdS;
    x = reinterpret_cast<__nv_bfloat16*>(dp + 16 * SM::kLdS);
    y = x + 16 * (kT + 8);
    float* rv = reinterpret_cast<float*>(base + 4 * size_t(SM::kTile) * 2 +
                                         kWarps * (2 * 16 * SM::kLdS * 4 + 2 * 16 * (kT + 8) * 2));
    lse = rv;
    dsum = rv + kT;
  }
};

// C (16 x 64, fp32, row stride ldc) = A (16 x D rows of a, row-major) .
// B^T where B is 64 x D rows of b (so B^T is b read column-major).
template <int D>
DEVI void mm_abt(float* c, int ldc, const __nv_bfloat16* a, const __nv_bfloat16* b) {
  constexpr int ld = Smem<D>::kLd;
#pragma unroll
  for (int n = 0; n < kT / 16; ++n) {
    wm::fragment<wm::accumulator, 16, 16, 16, float> acc;
    wm::fill_fragment(acc, 0.f);
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
      wm::fragment<wm::matrix_a, 16, 16, 16, __nv_bfloat16, wm::row_major> fa;
      wm::fragment<wm::matrix_b, 16, 16, 16, __nv_bfloat16, wm::col_major> fb;
      wm::load_matrix_sync(fa, a + kk * 16, ld);
      wm::load_matrix_sync(fb, b + n * 16 * ld + kk * 16, ld);
      wm::mma_sync(acc, fa, fb, acc);
    }
    wm::store_matrix_sync(c + n * 16, acc, ldc, wm::mem_row_major);
  }
}

// acc[n] (16 x 16 blocks of a 16 x D result) += X (16 x 64 bf16, row stride
// kT + 8) . T (64 x D rows of a shared tile, row-major).
template <int D>
DEVI void mm_acc(wm::fragment<wm::accumulator, 16, 16, 16, float> (&acc)[D / 16], const __nv_bfloat16* x,
                 const __nv_bfloat16* t) {
  constexpr int ld = Smem<D>::kLd;
#pragma unroll
  for (int kk = 0; kk < kT / 16; ++kk) {
    wm::fragment<wm::matrix_a, 16, 16, 16, __nv_bfloat16, wm::row_major> fa;
    wm::load_matrix_sync(fa, x + kk * 16, kT + 8);
#pragma unroll
    for (int n = 0; n < D / 16; ++n) {
      wm::fragment<wm::matrix_b, 16, 16, 16, __nv_bfloat16, wm::row_major> fb;
      wm::load_matrix_sync(fb, t + kk * 16 * ld + n * 16, ld);
      wm::mma_sync(acc[n], fa, fb, acc[n]);
    }
  }
}

// Writes scale * acc (16 x D) as bf16 rows row0.. (rows >= S skipped) of the
// [S, H, D] slice `head` of batch b, through the warp's fp32 S tile.
template <int D>
DEVI void store_rows(wm::fragment<wm::accumulator, 16, 16, 16, float> (&acc)[D / 16], float* stage, float scale,
                     __nv_bfloat16* dst, int b, int S, int H, int head, int row0) {
  constexpr int ldc = Smem<D>::kLdS;      // the 16 x 64 stage holds 64 columns at a time
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int half = 0; half < D / 64; ++half) {
#pragma unroll
    for (int n = 0; n < 4; ++n) wm::store_matrix_sync(stage + n * 16, acc[4 * half + n], ldc, wm::mem_row_major);
    __syncwarp();
    for (int e = lane; e < 16 * 64; e += 32) {
      const int r = e >> 6, c = e & 63;
      if (row0 + r < S)
        dst[((size_t(b) * S + row0 + r) * H + head) * D + 64 * half + c] = __float2bfloat16_rn(stage[r * ldc + c] * scale);
    }
    __syncwarp();
  }
}

template <int D>
__global__ void __launch_bounds__(kThreads) dq_kernel(const Params p) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  Carve<D> cv(smem, warp);
  __nv_bfloat16 *sQ = cv.t[0], *sdO = cv.t[1], *sK = cv.t[2], *sV = cv.t[3];
  const int q0 = blockIdx.x * kT, h = blockIdx.y, b = blockIdx.z, kvh = h / p.G;
  const int Lb = key_len(p, b);
  load_tile<D>(sQ, p.q, b, p.Sq, p.Hq, h, q0);
  load_tile<D>(sdO, p.dout, b, p.Sq, p.Hq, h, q0);
  for (int r = threadIdx.x; r < kT; r += kThreads) {
    const bool in = q0 + r < p.Sq;
    cv.lse[r] = in ? p.lse[(size_t(b) * p.Hq + h) * p.Sq + q0 + r] : 0.f;
    cv.dsum[r] = in ? p.dsum[(size_t(b) * p.Hq + h) * p.Sq + q0 + r] : 0.f;
  }
  // keys any row of the tile may see
  int kend = Lb;
  if (p.causal) kend = min(kend, min(q0 + kT, p.Sq) - 1 + p.Sk - p.Sq + 1);
  const int ntiles = kend > 0 ? (kend + kT - 1) / kT : 0;

  wm::fragment<wm::accumulator, 16, 16, 16, float> acc[D / 16];
#pragma unroll
  for (int n = 0; n < D / 16; ++n) wm::fill_fragment(acc[n], 0.f);
  const __nv_bfloat16* qw = sQ + warp * 16 * Smem<D>::kLd;
  const __nv_bfloat16* dow = sdO + warp * 16 * Smem<D>::kLd;
  for (int kt = 0; kt < ntiles; ++kt) {
    __syncthreads();
    load_tile<D>(sK, p.k, b, p.Sk, p.Hkv, kvh, kt * kT);
    load_tile<D>(sV, p.v, b, p.Sk, p.Hkv, kvh, kt * kT);
    __syncthreads();
    mm_abt<D>(cv.s, Smem<D>::kLdS, qw, sK);      // S = Q K^T
    mm_abt<D>(cv.dp, Smem<D>::kLdS, dow, sV);    // dP = dO V^T
    __syncwarp();
    for (int e = lane; e < 16 * kT; e += 32) {
      const int r = e >> 6, c = e & 63;
      const int i = q0 + warp * 16 + r, j = kt * kT + c;
      const bool ok = i < p.Sq && j < Lb && (!p.causal || j <= i + p.Sk - p.Sq);
      const float pr = ok ? __expf(cv.s[r * Smem<D>::kLdS + c] * p.scale - cv.lse[warp * 16 + r]) : 0.f;
      cv.x[r * (kT + 8) + c] =
          __float2bfloat16_rn(pr * (cv.dp[r * Smem<D>::kLdS + c] - cv.dsum[warp * 16 + r]));
    }
    __syncwarp();
    mm_acc<D>(acc, cv.x, sK);                    // dQ += dS K
  }
  store_rows<D>(acc, cv.s, p.scale, p.dq, b, p.Sq, p.Hq, h, q0 + warp * 16);
}

template <int D>
__global__ void __launch_bounds__(kThreads) dkdv_kernel(const Params p) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  Carve<D> cv(smem, warp);
  __nv_bfloat16 *sK = cv.t[0], *sV = cv.t[1], *sQ = cv.t[2], *sdO = cv.t[3];
  const int k0 = blockIdx.x * kT, kvh = blockIdx.y, b = blockIdx.z;
  const int Lb = key_len(p, b);
  load_tile<D>(sK, p.k, b, p.Sk, p.Hkv, kvh, k0);
  load_tile<D>(sV, p.v, b, p.Sk, p.Hkv, kvh, k0);
  // query rows that may see one of these keys: causal i >= k0 - (Sk - Sq)
  const int qfirst = (p.causal ? max(0, k0 - (p.Sk - p.Sq)) : 0) / kT;
  const int nq = (p.Sq + kT - 1) / kT;
  const bool any_key = k0 < Lb;

  wm::fragment<wm::accumulator, 16, 16, 16, float> dk[D / 16], dv[D / 16];
#pragma unroll
  for (int n = 0; n < D / 16; ++n) {
    wm::fill_fragment(dk[n], 0.f);
    wm::fill_fragment(dv[n], 0.f);
  }
  const __nv_bfloat16* kw = sK + warp * 16 * Smem<D>::kLd;
  const __nv_bfloat16* vw = sV + warp * 16 * Smem<D>::kLd;
  for (int g = 0; any_key && g < p.G; ++g) {
    const int h = kvh * p.G + g;
    for (int qt = qfirst; qt < nq; ++qt) {
      __syncthreads();
      load_tile<D>(sQ, p.q, b, p.Sq, p.Hq, h, qt * kT);
      load_tile<D>(sdO, p.dout, b, p.Sq, p.Hq, h, qt * kT);
      for (int r = threadIdx.x; r < kT; r += kThreads) {
        const bool in = qt * kT + r < p.Sq;
        cv.lse[r] = in ? p.lse[(size_t(b) * p.Hq + h) * p.Sq + qt * kT + r] : 0.f;
        cv.dsum[r] = in ? p.dsum[(size_t(b) * p.Hq + h) * p.Sq + qt * kT + r] : 0.f;
      }
      __syncthreads();
      mm_abt<D>(cv.s, Smem<D>::kLdS, kw, sQ);     // S^T = K Q^T (keys x queries)
      mm_abt<D>(cv.dp, Smem<D>::kLdS, vw, sdO);   // dP^T = V dO^T
      __syncwarp();
      for (int e = lane; e < 16 * kT; e += 32) {
        const int r = e >> 6, c = e & 63;
        const int j = k0 + warp * 16 + r, i = qt * kT + c;
        const bool ok = i < p.Sq && j < Lb && (!p.causal || j <= i + p.Sk - p.Sq);
        const float pr = ok ? __expf(cv.s[r * Smem<D>::kLdS + c] * p.scale - cv.lse[c]) : 0.f;
        cv.x[r * (kT + 8) + c] = __float2bfloat16_rn(pr);
        cv.y[r * (kT + 8) + c] = __float2bfloat16_rn(pr * (cv.dp[r * Smem<D>::kLdS + c] - cv.dsum[c]));
      }
      __syncwarp();
      mm_acc<D>(dv, cv.x, sdO);                   // dV += P^T dO
      mm_acc<D>(dk, cv.y, sQ);                    // dK += dS^T Q
    }
  }
  store_rows<D>(dk, cv.s, p.scale, p.dk, b, p.Sk, p.Hkv, kvh, k0 + warp * 16);
  store_rows<D>(dv, cv.s, 1.f, p.dv, b, p.Sk, p.Hkv, kvh, k0 + warp * 16);
}

}  // namespace bwd
}  // namespace gqa
