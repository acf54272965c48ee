// decode_fp8_sm103.cuh -- single-token GQA decode over an FP8 (e4m3) KV
// cache: the same split-KV method as decode_sm103.cuh with half the cache
// bytes.
//
// Sources (page title and section):
//  * GQA paper summary (azimuth.plus/paper/gqa), "Problem" / "Bottleneck":
//    a generation step reads the whole KV cache and is bound by memory
//    bandwidth; a smaller cache entry is a proportionally faster step.
//  * "3个GQA核心优化技巧" (blog.gitcode.com): quantisation named as a way to
//    compress the cache further; "阶段二" for split-KV (num_splits).
//  * "FlashAttention Serisi" (webturing.pages.dev), "Ana fikir": running
//    max / sum per split, partials merged through their log-sum-exp.
//
// Cache values are e4m3 with one scale per tensor: the attended key is
// k_scale * k8 and the value v_scale * v8.  Hence
//   s = scale * q.(k_scale k8) = (scale * k_scale) * q.k8
//   out = sum p v_scale v8 / l = v_scale * (sum p v8 / l)
// so k_scale folds into the softmax scale and v_scale into the output.
//
// CTA layout: one CTA per (split, group of kF8Warps K/V heads, b); warp w
// streams head kF8Warps * group + w over every 16-key block of the split
// through its own cp.async ring and writes that head's G output rows (or
// split partials) itself, so no warps are merged.  A cached row holds the
// Hkv heads side by side, so the CTA's warps read neighbouring 128-byte
// pieces of each row rather than one piece per CTA.
//
// Matrix products run on mma.sync m16n8k16 in f16: every e4m3 value is
// exact in f16 (cvt.rn.f16x2.e4m3x2), q is brought into f16's range by an
// exact power-of-two scaling 2^e of the whole group (2^-e folds into the
// score scale), and P in [0, 1] is held in f16.  Accumulation is fp32.
// Head dimension 128: a lane then reads exactly one 16-byte chunk of each
// of its four V rows per 16-key block.
#pragma once

#include "decode_sm103.cuh"

namespace gqa {
namespace decode {

constexpr int kF8D = 128;
constexpr int kF8Warps = 4;                 // warps per CTA = K/V heads per CTA
constexpr int kF8Threads = kF8Warps * 32;

struct ParamsF8 {
  const __nv_bfloat16* q;       // [B, Hq, 128]
  const uint8_t* kc;            // [B, Smax, Hkv, 128] e4m3
  const uint8_t* vc;            // [B, Smax, Hkv, 128] e4m3
  const int* seqlens;           // [B]
  __nv_bfloat16* out;           // [B, Hq, 128]         (nsplit == 1)
  float* part_o;                // [B, Hq, nsplit, 128] (nsplit > 1)
  float* part_lse;              // [B, Hq, nsplit]
  int B, Hq, Hkv, G, Smax;
  int nsplit, split_len;
  float scale_k_log2;           // scale * k_scale * log2(e)
  float v_scale;
};

// Per-warp ring of 16-key blocks, K rows then V rows, 128 bytes per row,
// chunks XOR-swizzled with swz() as in the bf16 ring.
struct RingF8 {
  static constexpr int kRing = 4;                          // 3 blocks in flight per warp, 3 CTAs (64 KB) per SM
  static constexpr uint32_t kRowBytes = kF8D;
  static constexpr uint32_t kSlotBytes = 2 * kBlockKeys * kRowBytes;
  static constexpr uint32_t kWarpBytes = kRing * kSlotBytes;
  static constexpr uint32_t kBytes = kF8Warps * kWarpBytes;
};

// two e4m3 values (low byte, high byte) -> f16x2 (low half, high half)
DEVI void e4m3x4_to_f16x2x2(uint32_t w, uint32_t& lo, uint32_t& hi) {
  asm("{\n\t.reg .b16 a, b;\n\tmov.b32 {a, b}, %2;\n\t"
      "cvt.rn.f16x2.e4m3x2 %0, a;\n\tcvt.rn.f16x2.e4m3x2 %1, b;\n}\n"
      : "=r"(lo), "=r"(hi)
      : "r"(w));
}

DEVI uint32_t pack_f16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

DEVI void mma_f16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                        uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Asynchronous copy of the 16-key block at key k0 into a ring slot; keys >=
// kend are zero-filled (source clamped to the valid row kvalid, 0 bytes read).
DEVI void issue_block_f8(uint32_t slot, const uint8_t* kbase, const uint8_t* vbase, size_t row_stride, int k0,
                         int kend, int kvalid, int lane) {
  constexpr int kChunks = kF8D / 16;
  constexpr int kPerLane = 2 * kBlockKeys * kChunks / 32;
#pragma unroll
  for (int i = 0; i < kPerLane; ++i) {
    const int id = lane + 32 * i;
    const int row = id / kChunks, chunk = id % kChunks;   // rows 0-15 K, 16-31 V
    const int key = k0 + (row & (kBlockKeys - 1));
    const bool ok = key < kend;
    const uint8_t* src = (row < kBlockKeys ? kbase : vbase) + size_t(ok ? key : kvalid) * row_stride + 16 * chunk;
    cp_async_16(slot + uint32_t(row) * RingF8::kRowBytes + (uint32_t(chunk) ^ swz(row)) * 16u, src, ok ? 16u : 0u);
  }
  cp_async_commit();
}

// Per-lane copy offsets of a 16-key block, fixed for the whole kernel: copy i
// of a lane moves 16-byte chunk (lane % 8) of row (lane / 8) + 4 (i % 4) of K
// (i < 4) or V (i >= 4).  goff: byte offset of that source chunk from the
// block's first cached row; soff: its swizzled place in the ring slot.
struct F8Copy {
  uint32_t goff[4];
  uint32_t soff[8];
};
DEVI F8Copy f8_copy_offsets(size_t row_stride, int lane) {
  F8Copy cp;
  const int chunk = lane & 7;
#pragma unroll
  for (int j = 0; j < 4; ++j) cp.goff[j] = uint32_t(((lane >> 3) + 4 * j) * row_stride) + 16u * uint32_t(chunk);
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int row = (i < 4 ? 0 : kBlockKeys) + (lane >> 3) + 4 * (i & 3);
    cp.soff[i] = uint32_t(row) * RingF8::kRowBytes + (uint32_t(chunk) ^ swz(row)) * 16u;
  }
  return cp;
}
// A block whose 16 keys are all valid: every copy moves 16 bytes.
DEVI void issue_full_block_f8(uint32_t slot, const uint8_t* kblk, const uint8_t* vblk, const F8Copy& cp) {
#pragma unroll
  for (int i = 0; i < 8; ++i)
    cp_async_16(slot + cp.soff[i], (i < 4 ? kblk : vblk) + cp.goff[i & 3], 16u);
  cp_async_commit();
}

// Raw e4m3 fragments of a block: K rows (r, r+8) chunks (c, c+4); V rows
// (2c, 2c+1, 2c+8, 2c+9) chunk r.
struct BlockF8 {
  uint4 k[2][2];
  uint4 v[4];
};

DEVI void fetch_block_f8(BlockF8& R, uint32_t slot, int r, int c) {
  constexpr uint32_t RB = RingF8::kRowBytes;
#pragma unroll
  for (int h = 0; h < 2; ++h)
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      const int row = r + 8 * h;
      R.k[h][q] = lds128(slot + uint32_t(row) * RB + (uint32_t(c + 4 * q) ^ swz(row)) * 16u);
    }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int row = kBlockKeys + 2 * c + (i & 1) + 8 * (i >> 1);
    R.v[i] = lds128(slot + uint32_t(row) * RB + (uint32_t(r) ^ swz(row)) * 16u);
  }
}

__global__ void __launch_bounds__(kF8Threads) decode_split_fp8_kernel(const ParamsF8 p) {
  constexpr int D = kF8D;
  constexpr int KS = D / 16;      // k-steps of QK^T
  constexpr int MT = D / 16;      // m-tiles of O^T
  const int split = blockIdx.x;
  const int b = blockIdx.z;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int r = lane >> 2;
  const int c = lane & 3;
  // warp w streams K/V head kvh = kF8Warps * blockIdx.y + w: the CTA's warps
  // read neighbouring 128-byte pieces of every cached row
  const int kvh = kF8Warps * int(blockIdx.y) + warp;
  if (kvh >= p.Hkv) return;

  int Lb = p.seqlens[b];
  if (Lb < 0 || Lb > p.Smax) {
    if (split == 0 && kvh == 0 && lane == 0) raise_error(kErrBounds);
    Lb = 0;
  }
  const int kstart = split * p.split_len;
  if (kstart >= Lb && p.nsplit > 1) return;  // empty split: the combine skips it
  const int kend = min(Lb, kstart + p.split_len);
  const int nblk = kend > kstart ? (kend - kstart + kBlockKeys - 1) / kBlockKeys : 0;

  const size_t row_stride = size_t(p.Hkv) * D;                       // bytes
  const uint8_t* kbase = p.kc + (size_t(b) * p.Smax * p.Hkv + kvh) * D;
  const uint8_t* vbase = p.vc + (size_t(b) * p.Smax * p.Hkv + kvh) * D;

  float o[MT][4];
#pragma unroll
  for (int mt = 0; mt < MT; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;
  float mA = -INFINITY, mB = -INFINITY, lA = 0.f, lB = 0.f;   // heads 2c and 2c+1

  // The ring prologue goes out before q is loaded and scaled, so the first
  // blocks' memory latency overlaps q's.
  using RG = RingF8;
  extern __shared__ __align__(16) uint8_t dsmem[];
  const uint32_t ring = smem_u32(dsmem) + uint32_t(warp) * RG::kWarpBytes;
  const F8Copy cpo = f8_copy_offsets(row_stride, lane);
  // a block of 16 valid keys takes the precomputed copy offsets; the
  // sequence's last, partial block zero-fills its keys past the end
  auto issue = [&](uint32_t slot, int k0) {
    if (k0 + kBlockKeys <= kend)
      issue_full_block_f8(slot, kbase + size_t(k0) * row_stride, vbase + size_t(k0) * row_stride, cpo);
    else
      issue_block_f8(slot, kbase, vbase, row_stride, k0, kend, kstart, lane);
  };
#pragma unroll
  for (int i = 0; i < RG::kRing - 1; ++i) {
    const int bi = i;
    if (bi < nblk)
      issue(ring + uint32_t(i) * RG::kSlotBytes, kstart + bi * kBlockKeys);
    else
      cp_async_commit();
  }
  // Q^T fragments (head n = r; zero if n >= G), dims d0..d0+3 of k-step ks
  // with d0 = 16 (c + 4 (ks / 4)) + 4 (ks % 4) -- the order in which the K
  // chunks below deliver them.  The whole group is scaled by 2^e so that its
  // largest |q| lies below 2^15 (exact; 2^-e goes into the score scale).
  float qv[KS][4];
  float qmax = 0.f;
  {
    const bool hv = r < p.G;
    const __nv_bfloat16* qrow = p.q + (size_t(b) * p.Hq + size_t(kvh) * p.G + (hv ? r : 0)) * D;
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
      const int d0 = 16 * (c + 4 * (ks >> 2)) + 4 * (ks & 3);
      const uint2 w = hv ? *reinterpret_cast<const uint2*>(qrow + d0) : make_uint2(0u, 0u);
      qv[ks][0] = __uint_as_float(w.x << 16);
      qv[ks][1] = __uint_as_float(w.x & 0xffff0000u);
      qv[ks][2] = __uint_as_float(w.y << 16);
      qv[ks][3] = __uint_as_float(w.y & 0xffff0000u);
#pragma unroll
      for (int e = 0; e < 4; ++e) qmax = fmaxf(qmax, fabsf(qv[ks][e]));
    }
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) qmax = fmaxf(qmax, __shfl_xor_sync(0xffffffffu, qmax, off));
  int ex = 0;
  if (qmax > 0.f && qmax < INFINITY) {
    frexpf(qmax, &ex);                     // qmax < 2^ex
    ex = max(-120, min(120, 15 - ex));     // 2^ex * qmax < 2^15
  }
  const float up = ldexpf(1.f, ex);
  uint32_t qf[KS][2];
#pragma unroll
  for (int ks = 0; ks < KS; ++ks) {
    qf[ks][0] = pack_f16x2(qv[ks][0] * up, qv[ks][1] * up);
    qf[ks][1] = pack_f16x2(qv[ks][2] * up, qv[ks][3] * up);
  }
  const float cl = p.scale_k_log2 * ldexpf(1.f, -ex);

  BlockF8 cur;
  int it = 0;
  for (int blk = 0; blk < nblk; ++blk, ++it) {
    cp_async_wait<RG::kRing - 2>();
    __syncwarp();
    fetch_block_f8(cur, ring + uint32_t(it % RG::kRing) * RG::kSlotBytes, r, c);
    __syncwarp();
    {
      const int nb = blk + (RG::kRing - 1);
      const uint32_t slot = ring + uint32_t((it + RG::kRing - 1) % RG::kRing) * RG::kSlotBytes;
      if (nb < nblk)
        issue(slot, kstart + nb * kBlockKeys);
      else
        cp_async_commit();
    }
    const int k0 = kstart + blk * kBlockKeys;

    // S^T = K . Q^T: k-step ks = 4 q + j uses raw word j of chunk c + 4q
    float s[4] = {0.f, 0.f, 0.f, 0.f}, s2[4] = {0.f, 0.f, 0.f, 0.f};   // two independent chains
#pragma unroll
    for (int q = 0; q < 2; ++q)
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        uint32_t a0, a2, a1, a3;
        e4m3x4_to_f16x2x2(word(cur.k[0][q], j), a0, a2);
        e4m3x4_to_f16x2x2(word(cur.k[1][q], j), a1, a3);
        if (j & 1)
          mma_f16_16816(s2, a0, a1, a2, a3, qf[4 * q + j][0], qf[4 * q + j][1]);
        else
          mma_f16_16816(s, a0, a1, a2, a3, qf[4 * q + j][0], qf[4 * q + j][1]);
      }
#pragma unroll
    for (int e = 0; e < 4; ++e) s[e] += s2[e];
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
    const uint32_t pb0 = movmatrix_trans(pack_f16x2(pA0, pB0));
    const uint32_t pb1 = movmatrix_trans(pack_f16x2(pA1, pB1));
    // O^T += V^T . P^T: m-tile mt rows r / r+8 are dims 16 r + 2 mt (+1),
    // taken from f16 word mt of each V row's chunk
#pragma unroll
    for (int wi = 0; wi < 4; ++wi) {
      uint32_t lo[4], hi[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) e4m3x4_to_f16x2x2(word(cur.v[i], wi), lo[i], hi[i]);
      mma_f16_16816(o[2 * wi], __byte_perm(lo[0], lo[1], 0x5410), __byte_perm(lo[0], lo[1], 0x7632),
                    __byte_perm(lo[2], lo[3], 0x5410), __byte_perm(lo[2], lo[3], 0x7632), pb0, pb1);
      mma_f16_16816(o[2 * wi + 1], __byte_perm(hi[0], hi[1], 0x5410), __byte_perm(hi[0], hi[1], 0x7632),
                    __byte_perm(hi[2], hi[3], 0x5410), __byte_perm(hi[2], hi[3], 0x7632), pb0, pb1);
    }
  }
  cp_async_wait<0>();

#pragma unroll
  for (int off = 4; off < 32; off <<= 1) {
    lA += __shfl_xor_sync(0xffffffffu, lA, off);
    lB += __shfl_xor_sync(0xffffffffu, lB, off);
  }

  // ---- this warp's G heads: lane (r, c) holds dims 16 r .. 16 r + 15 of
  // heads 2c and 2c+1 (o[mt][0 / 2]: dims 16 r + 2 mt / +1 of head 2c,
  // o[mt][1 / 3] of head 2c+1)
#pragma unroll
  for (int hh = 0; hh < 2; ++hh) {
    const int n = 2 * c + hh;
    if (n >= p.G) continue;
    const float l = hh ? lB : lA;
    const float m = hh ? mB : mA;
    const float inv = l > 0.f ? p.v_scale / l : 0.f;
    const size_t hrow = size_t(b) * p.Hq + size_t(kvh) * p.G + n;
    if (p.nsplit == 1) {
      uint32_t w[8];
#pragma unroll
      for (int mt = 0; mt < MT; ++mt) w[mt] = pack_bf16x2(o[mt][hh] * inv, o[mt][2 + hh] * inv);
      uint4* dst = reinterpret_cast<uint4*>(p.out + hrow * D + 16 * r);
      dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
      dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
    } else {
      float4* dst = reinterpret_cast<float4*>(p.part_o + (hrow * p.nsplit + split) * D + 16 * r);
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4)
        dst[q4] = make_float4(o[2 * q4][hh] * inv, o[2 * q4][2 + hh] * inv, o[2 * q4 + 1][hh] * inv,
                              o[2 * q4 + 1][2 + hh] * inv);
      if (r == 0) {
        float lg;
        asm("lg2.approx.f32 %0, %1;" : "=f"(lg) : "f"(l));
        p.part_lse[hrow * p.nsplit + split] = l > 0.f ? (m + lg) * 0.6931471805599453f : -INFINITY;
      }
    }
  }
}

}  // namespace decode
}  // namespace gqa
