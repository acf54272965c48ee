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
// 16-key blocks of the split (block w, w+4, ...).  K and V rows stream from
// global memory into a small per-warp shared-memory ring with 16-byte
// asynchronous copies (cp.async, one 16 B chunk = 8 consecutive head-dim
// values of one cached token), two or three blocks ahead of use, and are
// read from there directly in mma.sync fragment order:
//   S^T (16 keys x 8 heads) = K (16 x D) . Q^T (D x 8)   m16n8k16, K as A
//   O^T (D x 8 heads)      += V^T (D x 16) . P^T (16 x 8) m16n8k16, V^T as A
// The head-dimension index is permuted consistently between the K fragment
// and the Q fragment (a dot product does not depend on the order of its
// terms), and between the V fragment and the output rows.  P^T is formed
// from the S^T accumulator with movmatrix (an 8x8 transpose in registers).
// The work per byte is 8 flop/B, which would need ~52 TFLOP/s of fp32 FMA
// at full HBM bandwidth, hence the tensor cores.
#pragma once

#include <type_traits>

#include "common.cuh"

namespace gqa {
namespace decode {

constexpr int kWarps = 4;
constexpr int kThreads = kWarps * 32;
constexpr int kBlockKeys = 16;
constexpr float kRescaleThreshold = 8.0f;   // log2 units: p <= 2^8 (exact in bf16 and f16)

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

// Shared-memory ring of one warp: kRing slots, each one 16-key block of K
// rows then V rows, D*2 bytes per row.  The 16-byte chunk j of row `row` sits
// at chunk position j ^ swz(row): with it, each quarter-warp of the fragment
// reads below touches 8 distinct 16-byte bank groups (K: rows r, r+1 differ
// in bit 2 of the swizzle; V: rows 2c + x, c = 0..3, differ in bits 1-2).
template <int D>
struct Ring {
  static constexpr int kRing = (D == 128) ? 3 : 4;       // blocks per warp (in flight: kRing - 1)
  static constexpr uint32_t kRowBytes = D * 2;
  static constexpr uint32_t kSlotBytes = 2 * kBlockKeys * kRowBytes;
  static constexpr uint32_t kWarpBytes = kRing * kSlotBytes;
  static constexpr uint32_t kBytes = kWarps * kWarpBytes;   // dynamic shared memory per CTA
};

DEVI uint32_t swz(int row) { return uint32_t((((row >> 1) & 3) << 1) ^ ((row & 1) << 2)); }

// L2 policy for the cached K/V rows: each is read exactly once, so they are
// marked first to be evicted, which keeps the split partials (written during
// the kernel and read back by the combine) and q in L2 while gigabytes of
// cache stream through it.
DEVI uint64_t policy_evict_first() {
  uint64_t p;
  asm("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
DEVI void cp_async_16(uint32_t dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global.L2::cache_hint [%0], [%1], 16, %2, %3;" ::"r"(dst), "l"(src), "r"(src_bytes),
               "l"(policy_evict_first())
               : "memory");
}
DEVI void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
DEVI void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// Starts the asynchronous copy of the 16-key block at key k0 into ring slot
// `slot` (one commit group); keys >= kend are zero-filled (nothing is read
// for them: their source is clamped to a valid row and 0 bytes are copied).
template <int D>
DEVI void issue_block(uint32_t slot, const __nv_bfloat16* kbase, const __nv_bfloat16* vbase, size_t row_stride,
                      int k0, int kend, int kvalid, int lane) {
  constexpr int kChunks = D / 8;                    // 16-byte chunks per row
  constexpr int kPerLane = 2 * kBlockKeys * kChunks / 32;
#pragma unroll
  for (int i = 0; i < kPerLane; ++i) {
    const int id = lane + 32 * i;
    const int row = id / kChunks, chunk = id % kChunks;   // rows 0-15 K, 16-31 V
    const int key = k0 + (row & (kBlockKeys - 1));
    const bool ok = key < kend;
    const __nv_bfloat16* src = (row < kBlockKeys ? kbase : vbase) + size_t(ok ? key : kvalid) * row_stride + 8 * chunk;
    cp_async_16(slot + uint32_t(row) * Ring<D>::kRowBytes + (uint32_t(chunk) ^ swz(row)) * 16u, src, ok ? 16u : 0u);
  }
  cp_async_commit();
}

DEVI uint4 lds128(uint32_t a) {
  uint4 r;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "r"(a));
  return r;
}

// Fragments of a block from its ring slot, in mma.sync operand order:
// K rows (r, r+8) chunks c + 4q; V rows (2c, 2c+1, 2c+8, 2c+9) chunk 8 grp + r.
template <int D>
DEVI void fetch_block(BlockRegs<D>& R, uint32_t slot, int r, int c) {
  constexpr uint32_t RB = Ring<D>::kRowBytes;
#pragma unroll
  for (int h = 0; h < 2; ++h)
#pragma unroll
    for (int q = 0; q < D / 32; ++q) {
      const int row = r + 8 * h;
      R.k[h][q] = lds128(slot + uint32_t(row) * RB + (uint32_t(c + 4 * q) ^ swz(row)) * 16u);
    }
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int grp = 0; grp < D / 64; ++grp) {
      const int row = kBlockKeys + 2 * c + (i & 1) + 8 * (i >> 1);
      R.v[i][grp] = lds128(slot + uint32_t(row) * RB + (uint32_t(8 * grp + r) ^ swz(row)) * 16u);
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

  // This warp's blocks are warp, warp + 4, ...: kRing - 1 of them are always
  // on their way from global memory into the warp's ring while one is used.
  using RG = Ring<D>;
  extern __shared__ __align__(16) uint8_t dsmem[];
  const uint32_t ring = smem_u32(dsmem) + uint32_t(warp) * RG::kWarpBytes;
#pragma unroll
  for (int i = 0; i < RG::kRing - 1; ++i) {
    const int bi = warp + i * kWarps;
    if (bi < nblk)
      issue_block<D>(ring + uint32_t(i) * RG::kSlotBytes, kbase, vbase, row_stride, kstart + bi * kBlockKeys, kend,
                     kstart, lane);
    else
      cp_async_commit();     // keep one group per block position
  }
  BlockRegs<D> cur;
  int it = 0;
  for (int blk = warp; blk < nblk; blk += kWarps, ++it) {
    cp_async_wait<RG::kRing - 2>();
    __syncwarp();
    fetch_block<D>(cur, ring + uint32_t(it % RG::kRing) * RG::kSlotBytes, r, c);
    __syncwarp();            // every lane has read the slot refilled below (used one block ago)
    {
      const int nb = blk + (RG::kRing - 1) * kWarps;
      const uint32_t slot = ring + uint32_t((it + RG::kRing - 1) % RG::kRing) * RG::kSlotBytes;
      if (nb < nblk)
        issue_block<D>(slot, kbase, vbase, row_stride, kstart + nb * kBlockKeys, kend, kstart, lane);
      else
        cp_async_commit();
    }
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
    // The reference max of a head moves only when a block's max exceeds it by
    // more than kRescaleThreshold (log2 units), so p <= 2^threshold and O, l
    // are rescaled only then (a warp-uniform branch, rare after the first
    // blocks); the merge through the log-sum-exp is exact for any reference.
    const bool upA = xA > mA + kRescaleThreshold, upB = xB > mB + kRescaleThreshold;
    if (__any_sync(0xffffffffu, upA || upB)) {
      const float nA = upA ? xA : mA, nB = upB ? xB : mB;
      const float aA = (mA == -INFINITY) ? 0.f : ex2_approx(mA - nA);
      const float aB = (mB == -INFINITY) ? 0.f : ex2_approx(mB - nB);
      mA = nA;
      mB = nB;
      lA *= aA;
      lB *= aB;
#pragma unroll
      for (int mt = 0; mt < MT; ++mt) {
        o[mt][0] *= aA;
        o[mt][1] *= aB;
        o[mt][2] *= aA;
        o[mt][3] *= aB;
      }
    }
    const float rA = (mA == -INFINITY) ? 0.f : mA, rB = (mB == -INFINITY) ? 0.f : mB;
    const float pA0 = ex2_approx(tA0 - rA), pA1 = ex2_approx(tA1 - rA);
    const float pB0 = ex2_approx(tB0 - rB), pB1 = ex2_approx(tB1 - rB);
    lA += pA0 + pA1;
    lB += pB0 + pB1;
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
  }
  cp_async_wait<0>();

  // per-warp totals of l over the 8 lanes that share c
#pragma unroll
  for (int off = 4; off < 32; off <<= 1) {
    lA += __shfl_xor_sync(0xffffffffu, lA, off);
    lB += __shfl_xor_sync(0xffffffffu, lB, off);
  }

  // ---- combine the 4 warps through shared memory (the rings are done)
  __syncthreads();
  float (*s_o)[8][D] = reinterpret_cast<float (*)[8][D]>(dsmem);
  float (*s_m)[8] = reinterpret_cast<float (*)[8]>(dsmem + sizeof(float) * kWarps * 8 * D);
  float (*s_l)[8] = reinterpret_cast<float (*)[8]>(dsmem + sizeof(float) * (kWarps * 8 * D + kWarps * 8));
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
// and are skipped.  The lanes first reduce the split lse values and leave the
// normalised weights in shared memory; then each lane owns VEC consecutive
// head-dim values (VEC = D / 32 for D = 64 / 128, else a strided loop with
// VEC = 1) and reads every split's partial with independent vector loads.
// OutT is __nv_bfloat16 or float.
constexpr int kCombineMaxSplits = 128;

template <typename OutT, int VEC>
__global__ void __launch_bounds__(128)
    combine_kernel(const float* part_o, const float* part_lse, const int* seqlens, OutT* out,
                   int B, int Hq, int D, int nsplit, int split_len, int Smax) {
  __shared__ float s_w[4][kCombineMaxSplits];
  const int wib = threadIdx.x >> 5;
  const int row = blockIdx.x * 4 + wib;
  const int lane = threadIdx.x & 31;
  // Launched as a programmatic dependent of the split kernel: this grid may
  // start while the split kernel's last CTAs run, and waits here until that
  // grid has completed and its partials are visible.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if (row >= B * Hq) return;
  const int b = row / Hq;
  const float* lrow = part_lse + size_t(row) * nsplit;
  const float* orow = part_o + size_t(row) * nsplit * D;
  // Every load is issued before the key length (and with it the number of
  // splits that were written) is known, so that all their latencies overlap:
  // the first 32 splits' lse and the first kPre splits' partials.  Splits past
  // the sequence hold stale workspace values, which get no weight below.
  const float lse0 = lane < nsplit ? __ldcs(lrow + lane) : -INFINITY;
  constexpr int kPre = VEC > 1 ? 16 : 1;
  using V = typename std::conditional<VEC == 4, float4, float2>::type;
  V pre[kPre];
  if constexpr (VEC > 1) {
#pragma unroll
    for (int s = 0; s < kPre; ++s)
      if (s < nsplit) pre[s] = __ldcs(reinterpret_cast<const V*>(orow + size_t(s) * D) + lane);
  }
  int Lb = seqlens[b];
  if (Lb < 0 || Lb > Smax) Lb = 0;
  const int nvalid = min(min(nsplit, kCombineMaxSplits), (Lb + split_len - 1) / split_len);
  float M = -INFINITY;
  for (int s = lane; s < nvalid; s += 32) M = fmaxf(M, s < 32 ? lse0 : lrow[s]);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
  const float Mr = (M == -INFINITY) ? 0.f : M;
  float W = 0.f;
  for (int s = lane; s < nvalid; s += 32) {
    const float e = expf((s < 32 ? lse0 : lrow[s]) - Mr);
    s_w[wib][s] = e;
    W += e;
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) W += __shfl_xor_sync(0xffffffffu, W, off);
  __syncwarp();
  const float inv = W > 0.f ? 1.f / W : 0.f;
  if constexpr (VEC > 1) {
    // D == 32 * VEC: lane owns d = VEC*lane .. VEC*lane + VEC-1
    float acc[VEC];
#pragma unroll
    for (int e = 0; e < VEC; ++e) acc[e] = 0.f;
#pragma unroll
    for (int s = 0; s < kPre; ++s) {
      if (s < nvalid) {
        const V x = pre[s];
        const float w = s_w[wib][s];
        acc[0] += w * x.x;
        acc[1] += w * x.y;
        if constexpr (VEC == 4) {
          acc[2] += w * x.z;
          acc[3] += w * x.w;
        }
      }
    }
#pragma unroll 8
    for (int s = kPre; s < nvalid; ++s) {
      const V x = __ldcs(reinterpret_cast<const V*>(orow + size_t(s) * D) + lane);
      const float w = s_w[wib][s];
      acc[0] += w * x.x;
      acc[1] += w * x.y;
      if constexpr (VEC == 4) {
        acc[2] += w * x.z;
        acc[3] += w * x.w;
      }
    }
    OutT* o = out + size_t(row) * D + VEC * lane;
#pragma unroll
    for (int e = 0; e < VEC; ++e) {
      if constexpr (sizeof(OutT) == 2)
        o[e] = __float2bfloat16_rn(acc[e] * inv);
      else
        o[e] = acc[e] * inv;
    }
  } else {
    for (int d = lane; d < D; d += 32) {
      float acc = 0.f;
#pragma unroll 8
      for (int s = 0; s < nvalid; ++s) acc += s_w[wib][s] * __ldcs(orow + size_t(s) * D + d);
      const float val = acc * inv;
      if constexpr (sizeof(OutT) == 2)
        out[size_t(row) * D + d] = __float2bfloat16_rn(val);
      else
        out[size_t(row) * D + d] = val;
    }
  }
}

}  // namespace decode
}  // namespace gqa
