// backward_sm103.cuh -- gradients of the GQA forward (dQ, dK, dV), bf16, on
// the tcgen05 tensor cores with TMEM accumulators.
//
// Sources (page title and section): "FlashAttention Serisi"
// (webturing.pages.dev), "V2 katkısı" (a faster backward pass is one of its
// gains) and "Ana fikir" (the softmax intermediates stay out of slow memory;
// read here as: the weights are rebuilt from the forward's log-sum-exp,
// nothing quadratic is stored); "3个GQA核心优化技巧" (blog.gitcode.com),
// "GQA的分组共享机制": the G query heads of a group share one K/V head, so
// that head's gradient is the sum over the group.
//
// With P_ij = exp(scale q_i.k_j - lse_i) over the admissible keys (lse from
// the forward), Dsum_i = dO_i . O_i:
//   dV_j = sum_{h in group, i} P_ij dO_i
//   dS_ij = P_ij (dO_i . v_j - Dsum_i)
//   dQ_i = scale sum_j dS_ij k_j,   dK_j = scale sum_{h in group, i} dS_ij q_i
// Three kernels, no atomics, so the result does not depend on scheduling:
//  * dsum_kernel: Dsum per query row.
//  * dq_kernel, persistent (one CTA per SM claiming tiles), a tile being
//    Mq tokens x G heads of K/V head kvh = 128 rows (row = token * G +
//    head-in-group, as in the forward): per 128-key tile S = Q K^T and
//    dP = dO V^T into TMEM, dS = P (dP - Dsum) written back as packed bf16,
//    dQ += dS K accumulated in TMEM.
//  * dkdv_kernel, one CTA per (b, kvh, 128 keys): for every head of the group
//    and every query tile of 128, S^T = K Q^T and dP^T = V dO^T into TMEM,
//    P^T and dS^T written back over dP^T, dV += P^T dO and dK += dS^T Q
//    accumulated in TMEM over the whole loop (the group sum).
// Warp roles (576 threads): warps 0-15 the elementwise step and the
// epilogue, one TMEM lane (tile row) per thread and warp w taking the 32
// columns of group w / 4 of the row (four warps per SM sub-partition, so
// TMEM-load and MUFU latencies overlap), warp 16 TMA producer, warp 17 MMA
// issuer.  Tiles arrive by TMA with the 128-byte swizzle; the dq_kernel
// tile's Q and dO are copied into TMEM with tcgen05.cp and read from there
// as the A operand, which leaves the shared-memory operand bandwidth to the
// streamed K/V tiles.  All waits are bounded: on a timeout the kernel raises
// a device error, drains its copies and MMAs, and exits.
#pragma once

#include "common.cuh"

namespace gqa {
namespace bwd {

constexpr int kEwWarps = 16;             // elementwise warps: four per TMEM lane quarter
constexpr int kThreads = (kEwWarps + 2) * 32;
constexpr int kWarpTMA = kEwWarps;
constexpr int kWarpMMA = kEwWarps + 1;
constexpr int kBN = 128;                 // keys per tile (dq_kernel); keys per CTA (dkdv_kernel)
constexpr int kBQ = 128;                 // queries per tile (dkdv_kernel)
constexpr uint32_t kHalfBytes = 128u * 128u;   // 128 rows x 64 bf16 (128 bytes), one swizzle span
constexpr float kLog2e = 1.4426950408889634f;

struct Params {
  const __nv_bfloat16* o;       // [B, Sq, Hq, D]  forward output (dsum_kernel)
  const __nv_bfloat16* dout;    // [B, Sq, Hq, D]  (dsum_kernel)
  const float* lse;             // [B, Hq, Sq]     forward log-sum-exp (natural log)
  const int* seqlens;           // [B] or nullptr
  float* dsum;                  // [B, Hq, Sq]     Dsum, written by dsum_kernel
  __nv_bfloat16* dq;            // [B, Sq, Hq, D]
  __nv_bfloat16* dk;            // [B, Sk, Hkv, D]
  __nv_bfloat16* dv;            // [B, Sk, Hkv, D]
  int B, Hq, Hkv, G, Sq, Sk;
  int Mq;                       // tokens per dq_kernel tile (G * Mq <= 128)
  int n_qt;                     // dq_kernel tiles per (b, kvh): ceil(Sq / Mq)
  int n_kt;                     // dkdv_kernel tiles per (b, kvh): ceil(Sk / 128)
  int causal;
  float scale;
  float scale_log2;             // scale * log2(e)
  unsigned long long timeout_ns;
  // Test hook: when nonzero, the MMA issuer of dq_kernel and dkdv_kernel first
  // waits on its abort barrier, which nothing arrives on yet, so the wait runs
  // out after timeout_ns and the CTA takes its abort path.
  int test_stall;
  // dq_kernel's tile scheduler of this launch: sched[0] counts tiles claimed
  // past the first gridDim.x, sched[1] CTAs that finished; the last CTA to
  // finish sets both back to zero for the next launch that uses the slot.
  unsigned int* sched;
};

// Key length of batch entry b (a bad length raises a device error and
// counts as zero).
DEVI int key_len(const Params& p, int b) {
  int L = p.seqlens ? p.seqlens[b] : p.Sk;
  if (L < 0 || L > p.Sk) {
    raise_error(kErrBounds);
    L = 0;
  }
  return L;
}

// Dsum_i = dO_i . O_i: D / 8 consecutive threads per (b, h, i) row, each
// with one 16-byte load of dO and of O, reduced by shuffles.
template <int D>
__global__ void __launch_bounds__(256) dsum_kernel(const Params p) {
  constexpr int kTpr = D / 8;                     // threads per row (8 or 16)
  const long long nrows = (long long)p.B * p.Hq * p.Sq;
  const long long t = (long long)blockIdx.x * 256 + threadIdx.x;
  const long long row = t / kTpr;                 // row = (b * Sq + i) * Hq + h: memory order
  const int part = int(t % kTpr);
  float acc = 0.f;
  if (row < nrows) {
    const uint4 a = *reinterpret_cast<const uint4*>(p.dout + size_t(row) * D + part * 8);
    const uint4 o = *reinterpret_cast<const uint4*>(p.o + size_t(row) * D + part * 8);
    const uint32_t av[4] = {a.x, a.y, a.z, a.w}, ov[4] = {o.x, o.y, o.z, o.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 fa = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&av[e]));
      const float2 fo = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&ov[e]));
      acc = fmaf(fa.x, fo.x, acc);
      acc = fmaf(fa.y, fo.y, acc);
    }
  }
#pragma unroll
  for (int sh = kTpr / 2; sh > 0; sh >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, sh);
  if (row < nrows && part == 0) {
    const int h = int(row % p.Hq);
    const long long bi = row / p.Hq;              // b * Sq + i
    const int i = int(bi % p.Sq);
    const int b = int(bi / p.Sq);
    p.dsum[(size_t(b) * p.Hq + h) * p.Sq + i] = acc;
  }
}

// Shared-memory operand descriptors of a swizzled 128-row tile stored as
// 64-column halves of kHalfBytes each.
// K-major (the contraction runs along the tile's columns): 16-column step ks.
DEVI uint64_t desc_kmajor(uint32_t tile, int ks) {
  return make_sdesc_sw128(tile + uint32_t(ks / 4) * kHalfBytes + uint32_t(ks % 4) * 32u, 16, 1024);
}
// MN-major B (the contraction runs along the tile's rows, N along its
// columns): 16-row step ks; 8-row groups are 1024 bytes apart, and the second
// 64-column half (D = 128) is kHalfBytes further.
template <int D>
DEVI uint64_t desc_mnmajor(uint32_t tile, int ks) {
  return make_sdesc_sw128(tile + uint32_t(ks) * 2048u, D == 64 ? 1024u : kHalfBytes, 1024);
}
// Copies a K-major 128-row tile of D columns into TMEM columns
// [col, col + D/2) as packed bf16 pairs, the layout of a TMEM A operand.
template <int D>
DEVI void copy_tile_to_tmem(uint32_t tcol, uint32_t tile) {
#pragma unroll
  for (int ks = 0; ks < D / 16; ++ks) tmem_cp_128x256b(tcol + uint32_t(ks) * 8u, desc_kmajor(tile, ks));
}

// TMEM column of 16-key step ks of a bf16 operand written over a 128-column
// fp32 tile: the elementwise warps of column group c hold keys [32c, 32c+32)
// and write them as bf16 pairs into the first 16 of their own 32 columns.
DEVI uint32_t packed_col(int ks) { return uint32_t(ks / 2) * 32u + uint32_t(ks % 2) * 8u; }

// Writes 32 fp32 values times `mul` as bf16 to dst (16-byte aligned).
DEVI void store_row32(__nv_bfloat16* dst, const uint32_t* v, float mul) {
#pragma unroll
  for (int c8 = 0; c8 < 4; ++c8) {
    uint4 w;
    w.x = pack_bf16x2(__uint_as_float(v[8 * c8 + 0]) * mul, __uint_as_float(v[8 * c8 + 1]) * mul);
    w.y = pack_bf16x2(__uint_as_float(v[8 * c8 + 2]) * mul, __uint_as_float(v[8 * c8 + 3]) * mul);
    w.z = pack_bf16x2(__uint_as_float(v[8 * c8 + 4]) * mul, __uint_as_float(v[8 * c8 + 5]) * mul);
    w.w = pack_bf16x2(__uint_as_float(v[8 * c8 + 6]) * mul, __uint_as_float(v[8 * c8 + 7]) * mul);
    *reinterpret_cast<uint4*>(dst + 8 * c8) = w;
  }
}
DEVI void store_zero_row(__nv_bfloat16* dst, int n) {
  for (int c = 0; c < n; c += 8) *reinterpret_cast<uint4*>(dst + c) = make_uint4(0u, 0u, 0u, 0u);
}

// ------------------------------------------------------------------ dq_kernel
template <int D>
struct DqLayout {
  static constexpr int kHalves = D / 64;
  static constexpr uint32_t kTileBytes = kHalves * kHalfBytes;
  static constexpr int kStages = (D == 64) ? 3 : 2;        // K/V ring depth
  static constexpr uint32_t kOffQ = 0;
  static constexpr uint32_t kOffDO = kTileBytes;
  static constexpr uint32_t kOffK = 2 * kTileBytes;
  static constexpr uint32_t kOffV = kOffK + kStages * kTileBytes;
  static constexpr uint32_t kOffBar = kOffV + kStages * kTileBytes;
  // q_full, kv_full[S], kv_empty[S], s_full, p_full, done, drain, sd_read, dq_done, q_empty, dq_free,
  // tq_full[kTQ], tq_empty[kTQ]
  static constexpr int kTQ = 4;                            // tile-queue entries
  static constexpr int kNumBars = 1 + 2 * kStages + 8 + 2 * kTQ;
  static constexpr uint32_t kOffTQ = kOffBar + 8u * kNumBars;   // [kTQ] int: claimed tile indices
  static constexpr uint32_t kOffSlot = kOffTQ + 4u * kTQ;
  static constexpr uint32_t kOffAbort = kOffSlot + 8u;
  static constexpr uint32_t kBytes = kOffAbort + 8u;
  static constexpr uint32_t kSmemAlloc = kBytes + 1024u;
  // TMEM: S [0,128), dP [128,256), Q [256, 256+D/2), dO [256+D/2, 256+D),
  // dQ [256+D, 256+2D).  dS (bf16 pairs): D = 64 in its own columns
  // [384, 448), so that S and dP are free as soon as they have been read;
  // D = 128 over dP, column group c's 32 keys in [128 + 32c, 128 + 32c + 16).
  static constexpr bool kSepDS = (D == 64);
  static constexpr uint32_t kTmS = 0, kTmP = 128, kTmQ = 256, kTmDO = 256 + D / 2, kTmDQ = 256 + D;
  static constexpr uint32_t kTmDS = 256 + 2 * D;
  static constexpr uint32_t kTmCols = 512;
  static_assert(kTmDQ + D <= kTmCols, "TMEM column map overflows");
  static_assert(!kSepDS || kTmDS + 64 <= kTmCols, "TMEM column map overflows");
  static_assert(kSmemAlloc > 116u * 1024u, "one CTA per SM: its TMEM allocation takes all 512 columns");
};

// ---------------------------------------------------------------- dkdv_kernel
template <int D>
struct KvLayout {
  static constexpr int kHalves = D / 64;
  static constexpr uint32_t kTileBytes = kHalves * kHalfBytes;
  static constexpr int kStages = (D == 64) ? 3 : 2;        // Q/dO ring depth
  static constexpr int kDPBufs = (D == 64) ? 2 : 1;        // dP^T buffers in TMEM
  static constexpr uint32_t kOffK = 0;
  static constexpr uint32_t kOffV = kTileBytes;
  static constexpr uint32_t kOffQ = 2 * kTileBytes;
  static constexpr uint32_t kOffDO = kOffQ + kStages * kTileBytes;
  static constexpr uint32_t kOffRow = kOffDO + kStages * kTileBytes;   // [2][2][128] fp32: -lse*log2e, -Dsum
  static constexpr uint32_t kOffBar = kOffRow + 2u * 2u * kBQ * 4u;
  // kv_full, qd_full[S], qd_empty[S], s_full, p_full[0], done, drain, row_full[2], sd_read, p_full[1]
  static constexpr int kNumBars = 1 + 2 * kStages + 4 + 2 + 1 + 1;
  static constexpr uint32_t kOffSlot = kOffBar + 8u * kNumBars;
  static constexpr uint32_t kOffAbort = kOffSlot + 8u;
  static constexpr uint32_t kBytes = kOffAbort + 8u;
  static constexpr uint32_t kSmemAlloc = kBytes + 1024u;
  // TMEM: S^T [0,128), dP^T buffer 0 [128,256), dV [256, 256+D), dK
  // [256+D, 256+2D), and at D = 64 dP^T buffer 1 [384,512).  The bf16 pairs
  // of column group c's 32 queries go over that group's columns of the dP^T
  // buffer they were computed in: dS^T in [+32c, +16), P^T in [+32c+16, +16).
  // S^T is free as soon as it has been read; with two dP^T buffers the next
  // iteration's dP^T goes into the other one while dV and dK still read this.
  static constexpr uint32_t kTmS = 0, kTmDV = 256, kTmDK = 256 + D;
  static constexpr uint32_t kTmP0 = 128, kTmP1 = (kDPBufs == 2) ? 384 : 128;
  static constexpr uint32_t kTmCols = 512;
  static_assert(kTmDK + D <= kTmCols && (kDPBufs == 1 || kTmDK + D <= kTmP1), "TMEM column map overflows");
  static_assert(kSmemAlloc > 116u * 1024u, "one CTA per SM: its TMEM allocation takes all 512 columns");
};

// dQ, persistent: CTA c takes tile c first, then claims tiles from a
// counter in global memory (dynamic scheduling: it runs beside dkdv_kernel,
// whose CTAs leave SMs at different times), out of the n_qt * Hkv * B tiles
// (tile = Mq tokens x G heads of K/V head kvh, batch b; the token block varies
// fastest, so CTAs running at one time share K/V in L2).
// Iteration counters run on across tiles, so the next tile's Q/dO and K/V
// land while the current one is computed.  Schedule over a tile's key tiles
// j (one issuing thread: the tensor core runs its MMAs in issue order):
//   issuer:      S(0), dP(0); then per j: once the elementwise warps have read
//                S(j) and dP(j): S(j+1) (and dP(j+1) when dS has its own
//                columns); once dS(j) is written: dQ += dS(j) K(j) (then
//                dP(j+1) when dS lies over dP).  A tile's first dQ waits for
//                the previous tile's epilogue to have read dQ.
//   elementwise: per j: read S(j), dP(j); signal; dS(j) = P (dP - Dsum) in
//                registers; write dS(j) (its own columns: after the previous
//                dQ product has read them); signal.  Then the epilogue.
template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    dq_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmDO,
              const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV, const Params p) {
  using L = DqLayout<D>;
  constexpr int S = L::kStages;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  const uint32_t base = (raw_addr + 1023u) & ~1023u;
  uint8_t* sbase = smem_raw + (base - raw_addr);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  auto bar = [&](int i) -> uint32_t { return base + L::kOffBar + 8u * uint32_t(i); };
  const uint32_t q_full = bar(0);
  auto kv_full = [&](int s) { return bar(1 + s); };
  auto kv_empty = [&](int s) { return bar(1 + S + s); };
  const uint32_t s_full = bar(1 + 2 * S), p_full = bar(2 + 2 * S), done = bar(3 + 2 * S), drain = bar(4 + 2 * S);
  const uint32_t sd_read = bar(5 + 2 * S), dq_done = bar(6 + 2 * S);
  const uint32_t q_empty = bar(7 + 2 * S), dq_free = bar(8 + 2 * S);
  auto tq_full = [&](int i) { return bar(9 + 2 * S + i); };
  auto tq_empty = [&](int i) { return bar(9 + 2 * S + L::kTQ + i); };
  volatile int* tq = reinterpret_cast<volatile int*>(sbase + L::kOffTQ);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sbase + L::kOffAbort);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sbase + L::kOffSlot);
  const uint64_t to = p.timeout_ns;
  const int n_tiles = p.n_qt * p.Hkv * p.B;
  const int diag = p.Sk - p.Sq;               // causal: query i sees keys j <= i + diag

  // tile -> (batch, K/V head, first token, key length, number of key tiles)
  struct Tile {
    int b, kvh, q0, Lb, n;
  };
  auto tile_info = [&](int t) -> Tile {
    Tile T;
    const int x = t % p.n_qt;
    const int rest = t / p.n_qt;
    T.kvh = rest % p.Hkv;
    T.b = rest / p.Hkv;
    T.q0 = x * p.Mq;
    T.Lb = key_len(p, T.b);
    int kmax = T.Lb;
    if (p.causal) kmax = min(kmax, min(T.q0 + p.Mq, p.Sq) - 1 + diag + 1);
    T.n = kmax > 0 ? (kmax + kBN - 1) / kBN : 0;
    return T;
  };
  // Tiles are claimed at run time: the producer publishes this CTA's kq-th
  // tile (blockIdx.x first, then claims from the launch's counter, one tile
  // ahead) in queue entry kq % kTQ; n_tiles or more ends the loops.  A warp
  // (elementwise) releases the entry with one arrival once every lane has
  // read it; the MMA thread arrives itself.
  auto next_tile = [&](int kq, bool& okq, bool whole_warp) -> int {
    const int qi = kq % L::kTQ;
    okq = mbar_wait(tq_full(qi), (kq / L::kTQ) & 1, abort_flag, p.timeout_ns);
    const int t = okq ? tq[qi] : n_tiles;
    if (whole_warp) {
      __syncwarp();
      if ((threadIdx.x & 31) == 0) mbar_arrive(tq_empty(qi));
    } else {
      mbar_arrive(tq_empty(qi));
    }
    return t;
  };

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    mbar_init(q_empty, 1);
    for (int s = 0; s < S; ++s) {
      mbar_init(kv_full(s), 1);
      mbar_init(kv_empty(s), 1);
    }
    mbar_init(s_full, 1);
    mbar_init(p_full, kEwWarps);   // one arrival per elementwise warp
    mbar_init(done, 1);
    mbar_init(drain, 1);
    mbar_init(sd_read, kEwWarps);
    mbar_init(dq_done, 1);
    mbar_init(dq_free, kEwWarps);
    for (int i = 0; i < L::kTQ; ++i) {
      mbar_init(tq_full(i), 1);
      mbar_init(tq_empty(i), 1 + kEwWarps);   // the MMA thread and one arrival per elementwise warp
    }
    *abort_flag = 0;
    fence_mbar_init();
    fence_proxy_async_smem();
  }
  if (warp == kWarpMMA) {
    tmem_alloc(smem_u32(tmem_slot), L::kTmCols);
    tmem_relinquish();
  }
  if (warp == kWarpTMA && lane == 0) {
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmDO);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == kWarpTMA) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const uint32_t q_bytes = 2u * uint32_t(L::kHalves) * 128u * uint32_t(p.G * p.Mq);
      bool ok = true;
      int g = 0;                  // K/V tiles loaded so far (ring position)
      int k = 0;                  // tiles with work so far (Q/dO buffer phase)
      int t_next = int(blockIdx.x);
      for (int kq = 0; ok; ++kq) {
        const int t = t_next;
        const int qi = kq % L::kTQ;
        ok = mbar_wait(tq_empty(qi), ((kq / L::kTQ) & 1) ^ 1, abort_flag, to);
        if (!ok) break;
        if (t < n_tiles) {
          unsigned int v;
          asm volatile("atom.global.add.u32 %0, [%1], 1;" : "=r"(v) : "l"(p.sched) : "memory");
          t_next = int(gridDim.x + v);
        }
        tq[qi] = t;
        mbar_arrive(tq_full(qi));   // release: the entry is visible to the consumers
        if (t >= n_tiles) break;
        const Tile T = tile_info(t);
        if (T.n == 0) continue;
        // the Q/dO buffer is free once the previous tile's copies into TMEM are done
        ok = mbar_wait(q_empty, (k & 1) ^ 1, abort_flag, to);
        if (!ok) break;
        mbar_arrive_expect_tx(q_full, q_bytes);
        for (int hh = 0; hh < L::kHalves; ++hh) {
          tma_load_4d(base + L::kOffQ + hh * kHalfBytes, &tmQ, q_full, hh * 64, T.kvh * p.G, T.q0, T.b);
          tma_load_4d(base + L::kOffDO + hh * kHalfBytes, &tmDO, q_full, hh * 64, T.kvh * p.G, T.q0, T.b);
        }
        ++k;
        for (int j = 0; j < T.n; ++j, ++g) {
          const int s = g % S;
          ok = mbar_wait(kv_empty(s), ((g / S) & 1) ^ 1, abort_flag, to);
          if (!ok) break;
          mbar_arrive_expect_tx(kv_full(s), 2u * L::kTileBytes);
          for (int hh = 0; hh < L::kHalves; ++hh) {
            tma_load_4d(base + L::kOffK + s * L::kTileBytes + hh * kHalfBytes, &tmK, kv_full(s), hh * 64,
                        T.kvh, j * kBN, T.b);
            tma_load_4d(base + L::kOffV + s * L::kTileBytes + hh * kHalfBytes, &tmV, kv_full(s), hh * 64,
                        T.kvh, j * kBN, T.b);
          }
        }
      }
      if (!ok) {
        // let the copies in flight land before the CTA exits: each waited
        // phase belongs to the last load issued into its buffer
        volatile int no_abort = 0;
        for (int it = g > S ? g - S : 0; it < g; ++it)
          mbar_wait(kv_full(it % S), (it / S) & 1, &no_abort, 200000000ull);
        if (k > 0) mbar_wait(q_full, (k - 1) & 1, &no_abort, 200000000ull);
      }
    }
  } else if (warp == kWarpMMA) {
    // ---------------------------------------------------------- MMA issuer
    if (lane == 0) {
      const uint32_t idesc_s = make_idesc_bf16(128, kBN, 0, 0);   // A in TMEM, B K-major
      const uint32_t idesc_q = make_idesc_bf16(128, D, 0, 1);     // dS in TMEM, K MN-major
      auto issue_s = [&](int it) {          // S = Q K^T, K from ring stage it % S
        const uint32_t ka = base + L::kOffK + (it % S) * L::kTileBytes;
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks)
          umma_ts(tmem + L::kTmS, tmem + L::kTmQ + uint32_t(ks) * 8u, desc_kmajor(ka, ks), idesc_s,
                  ks > 0 ? 1u : 0u);
      };
      auto issue_dp = [&](int it) {         // dP = dO V^T
        const uint32_t va = base + L::kOffV + (it % S) * L::kTileBytes;
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks)
          umma_ts(tmem + L::kTmP, tmem + L::kTmDO + uint32_t(ks) * 8u, desc_kmajor(va, ks), idesc_s,
                  ks > 0 ? 1u : 0u);
      };
      // test hook: `drain` has no arrival yet
      bool ok = !p.test_stall || mbar_wait(drain, 0, abort_flag, to);
      int g = 0;                  // key-tile iterations so far (all tiles)
      int k = 0;                  // tiles with work so far
      for (int kq = 0; ok; ++kq) {
        const int t = next_tile(kq, ok, false);
        if (!ok || t >= n_tiles) break;
        const int n = tile_info(t).n;
        if (n == 0) continue;
        ok = mbar_wait(q_full, k & 1, abort_flag, to) && mbar_wait(kv_full(g % S), (g / S) & 1, abort_flag, to);
        if (!ok) break;
        tc_fence_after();
        // executes after every MMA issued before it, so the previous tile's
        // S and dP products have read the old Q and dO
        copy_tile_to_tmem<D>(tmem + L::kTmQ, base + L::kOffQ);
        copy_tile_to_tmem<D>(tmem + L::kTmDO, base + L::kOffDO);
        umma_commit(q_empty);
        issue_s(g);
        issue_dp(g);
        umma_commit(s_full);
        for (int j = 0; ok && j < n; ++j) {
          const int it = g + j;
          const bool more = j + 1 < n;
          // S(j) and dP(j) have been read: S(j+1) (and dP(j+1)) may overwrite them
          ok = mbar_wait(sd_read, it & 1, abort_flag, to);
          if (ok && more) ok = mbar_wait(kv_full((it + 1) % S), ((it + 1) / S) & 1, abort_flag, to);
          if (!ok) break;
          tc_fence_after();
          if (more) {
            issue_s(it + 1);
            if constexpr (L::kSepDS) {
              issue_dp(it + 1);
              umma_commit(s_full);
            }
          }
          ok = mbar_wait(p_full, it & 1, abort_flag, to);
          // the tile's first dQ product overwrites dQ: the previous epilogue must have read it
          if (ok && j == 0 && k > 0) ok = mbar_wait(dq_free, (k - 1) & 1, abort_flag, to);
          if (!ok) break;
          tc_fence_after();
          // dQ += dS(j) K(j)
          const uint32_t ka = base + L::kOffK + (it % S) * L::kTileBytes;
#pragma unroll
          for (int ks = 0; ks < kBN / 16; ++ks) {
            const uint32_t acol = L::kSepDS ? L::kTmDS + uint32_t(ks) * 8u : L::kTmP + packed_col(ks);
            umma_ts(tmem + L::kTmDQ, tmem + acol, desc_mnmajor<D>(ka, ks), idesc_q, (j > 0 || ks > 0) ? 1u : 0u);
          }
          umma_commit(kv_empty(it % S));
          if constexpr (L::kSepDS) {
            umma_commit(dq_done);
          } else if (more) {
            issue_dp(it + 1);               // dP(j+1) over dS(j), after dQ has read it
            umma_commit(s_full);
          }
        }
        if (!ok) break;
        umma_commit(done);
        g += n;
        ++k;
      }
      if (!ok) {
        volatile int no_abort = 0;
        umma_commit(drain);
        mbar_wait(drain, 0, &no_abort, 200000000ull);
      }
    }
  } else {
    // ------------------------------------------------- elementwise + epilogue
    // warp w: TMEM lanes 32 (w % 4) .. +31 (tile rows), keys of column group w / 4
    const int r = (warp & 3) * 32 + lane;
    const int grp = warp >> 2;
    const uint32_t lane_base = uint32_t((warp & 3) * 32) << 16;
    const int token = r / p.G, gg = r - token * p.G;
    const uint64_t cl2 = f2_pack(p.scale_log2, p.scale_log2);
    // where this group's dS goes (bf16 pairs, 16 columns)
    const uint32_t ds_col = L::kSepDS ? L::kTmDS + uint32_t(grp) * 16u : L::kTmP + uint32_t(grp) * 32u;
    bool aborted = false;
    int g = 0;                    // key-tile iterations so far (all tiles)
    int k = 0;                    // tiles with work so far
    for (int kq = 0; !aborted; ++kq) {
      bool okq;
      const int t = next_tile(kq, okq, true);
      if (!__all_sync(0xffffffffu, okq)) {
        aborted = true;
        break;
      }
      if (t >= n_tiles) break;
      const Tile T = tile_info(t);
      const int i = T.q0 + token;
      const bool row_ok = r < p.G * p.Mq && i < p.Sq;
      const int h = T.kvh * p.G + gg;
      __nv_bfloat16* drow = p.dq + ((size_t(T.b) * p.Sq + i) * p.Hq + h) * D + grp * 32;
      if (T.n == 0) {
        if (row_ok && grp < D / 32) store_zero_row(drow, 32);    // no admissible key: dQ = 0
        continue;
      }
      const size_t rowidx = (size_t(T.b) * p.Hq + h) * p.Sq + i;
      float lse2 = 0.f, dsum = 0.f;
      int hi_row = 0;                                   // the row admits keys j < hi_row
      if (row_ok) {
        lse2 = p.lse[rowidx] * kLog2e;
        dsum = p.dsum[rowidx];
        hi_row = p.causal ? min(T.Lb, i + diag + 1) : T.Lb;
      }
      const uint64_t nl2 = f2_pack(-lse2, -lse2);
      const uint64_t nd2 = f2_pack(-dsum, -dsum);
      for (int j = 0; j < T.n; ++j) {
        const int it = g + j;
        bool ok = __all_sync(0xffffffffu, mbar_wait(s_full, it & 1, abort_flag, to));
        if (!ok) {
          aborted = true;
          break;
        }
        tc_fence_after();
        // this warp's 32 keys of the tile: [grp * 32, grp * 32 + 32)
        const int lim = hi_row - j * kBN - grp * 32;
        const bool full = __all_sync(0xffffffffu, lim >= 32 || !row_ok);
        // two 16-key chunks through the same registers; S and dP are free for
        // the next products once the second chunk is in registers
        uint32_t sv[16], dp[16], ds[16];
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          tmem_ld_32x32b_x16(tmem + lane_base + L::kTmS + uint32_t(grp) * 32u + uint32_t(c) * 16u, sv);
          tmem_ld_32x32b_x16(tmem + lane_base + L::kTmP + uint32_t(grp) * 32u + uint32_t(c) * 16u, dp);
          tmem_ld_wait_x16(sv);
          tmem_ld_wait_x16(dp);
          if (c == 1) {
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(sd_read);
          }
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const int k0 = 16 * c + 2 * e;
            float x0, x1, p0, p1, t0, t1;
            f2_unpack(f2_fma(f2_pack(__uint_as_float(sv[2 * e]), __uint_as_float(sv[2 * e + 1])), cl2, nl2), x0,
                      x1);
            p0 = ex2_approx(x0);
            p1 = ex2_approx(x1);
            if (!full) {
              p0 = (k0 < lim) ? p0 : 0.f;
              p1 = (k0 + 1 < lim) ? p1 : 0.f;
            }
            f2_unpack(f2_add(f2_pack(__uint_as_float(dp[2 * e]), __uint_as_float(dp[2 * e + 1])), nd2), t0, t1);
            ds[8 * c + e] = pack_bf16x2(p0 * t0, p1 * t1);
          }
        }
        if (L::kSepDS && it > 0) {
          // the previous dQ product must have read the dS columns
          ok = __all_sync(0xffffffffu, mbar_wait(dq_done, (it - 1) & 1, abort_flag, to));
          if (!ok) {
            aborted = true;
            break;
          }
          tc_fence_after();
        }
        tmem_st_32x32b_x16(tmem + lane_base + ds_col, ds);
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(p_full);
      }
      if (aborted) break;
      // epilogue: column group grp < D / 32 writes dQ columns [32 grp, 32 grp + 32)
      const bool ok = __all_sync(0xffffffffu, mbar_wait(done, k & 1, abort_flag, to));
      if (!ok) {
        aborted = true;
        break;
      }
      tc_fence_after();
      uint32_t v[32];
      if (grp < D / 32) {
        tmem_ld_32x32b_x32(tmem + lane_base + L::kTmDQ + uint32_t(grp) * 32u, v);
        tmem_ld_wait_x32(v);
      }
      // dQ has been read: the next tile's first product may overwrite it
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(dq_free);
      if (row_ok && grp < D / 32) store_row32(drow, v, p.scale);
      g += T.n;
      ++k;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kWarpMMA) {
    tc_fence_after();
    tmem_dealloc(tmem, L::kTmCols);
  }
  if (threadIdx.x == 0) {
    // every claim of this CTA is done: count it out; the last CTA resets the
    // scheduler slot for the next launch that uses it
    __threadfence();
    if (atomicAdd(p.sched + 1, 1u) == gridDim.x - 1) {
      atomicExch(p.sched, 0u);
      atomicExch(p.sched + 1, 0u);
    }
  }
}

// dK and dV for 128 keys of K/V head kvh, batch b.  Iteration it covers head
// kvh * G + it / nqe of the group and query tile qfirst + it % nqe.
//   issuer:      S^T(0), dP^T(0); then per it: once the elementwise warps
//                have read S^T(it) and dP^T(it): S^T(it+1) (and with two dP^T
//                buffers dP^T(it+1) into the other one); once P^T(it) and
//                dS^T(it) are written (over dP^T(it)): dV += P^T dO,
//                dK += dS^T Q (then, with one buffer, dP^T(it+1): issue order
//                keeps it behind their reads)
//   elementwise: per it: read S^T(it), dP^T(it); signal; P^T, dS^T in
//                registers; write them over dP^T(it); signal
// so the next scores are computed while the elementwise warps work on
// iteration it and, with two buffers, dV and dK overlap the next iteration.
template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    dkdv_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmDO, const Params p) {
  using L = KvLayout<D>;
  constexpr int S = L::kStages;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  const uint32_t base = (raw_addr + 1023u) & ~1023u;
  uint8_t* sbase = smem_raw + (base - raw_addr);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  auto bar = [&](int i) -> uint32_t { return base + L::kOffBar + 8u * uint32_t(i); };
  const uint32_t kv_full = bar(0);
  auto qd_full = [&](int s) { return bar(1 + s); };
  auto qd_empty = [&](int s) { return bar(1 + S + s); };
  const uint32_t s_full = bar(1 + 2 * S), done = bar(3 + 2 * S), drain = bar(4 + 2 * S);
  auto row_full = [&](int i) { return bar(5 + 2 * S + i); };
  const uint32_t sd_read = bar(7 + 2 * S);
  // p_full for iteration it is barrier it & 1: an iteration's arrivals never
  // meet the previous one's on the same barrier before the issuer has seen it
  auto p_full = [&](int i) { return i ? bar(8 + 2 * S) : bar(2 + 2 * S); };
  auto tm_dp = [&](int it) -> uint32_t { return (L::kDPBufs == 2 && (it & 1)) ? L::kTmP1 : L::kTmP0; };
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sbase + L::kOffAbort);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sbase + L::kOffSlot);
  float* rowv = reinterpret_cast<float*>(sbase + L::kOffRow);   // [2][2][kBQ]: -lse * log2(e), -Dsum
  const uint64_t to = p.timeout_ns;

  const int kvh = blockIdx.y, b = blockIdx.z;
  const int k0 = blockIdx.x * kBN;
  const int Lb = key_len(p, b);
  const int diag = p.Sk - p.Sq;               // causal: query i sees keys j <= i + diag
  const int nq = (p.Sq + kBQ - 1) / kBQ;
  // causal: the first query that sees key k0 is k0 - diag
  const int qfirst = p.causal ? max(0, k0 - diag) / kBQ : 0;
  const int nqe = (k0 < Lb && qfirst < nq) ? nq - qfirst : 0;
  const int n = p.G * nqe;

  if (threadIdx.x == 0) {
    mbar_init(kv_full, 1);
    for (int s = 0; s < S; ++s) {
      mbar_init(qd_full(s), 1);
      mbar_init(qd_empty(s), 1);
    }
    mbar_init(s_full, 1);
    mbar_init(p_full(0), kEwWarps);   // one arrival per elementwise warp
    mbar_init(p_full(1), kEwWarps);
    mbar_init(done, 1);
    mbar_init(drain, 1);
    mbar_init(row_full(0), kEwWarps);
    mbar_init(row_full(1), kEwWarps);
    mbar_init(sd_read, kEwWarps);
    *abort_flag = 0;
    fence_mbar_init();
    fence_proxy_async_smem();
  }
  if (warp == kWarpMMA) {
    tmem_alloc(smem_u32(tmem_slot), L::kTmCols);
    tmem_relinquish();
  }
  if (warp == kWarpTMA && lane == 0) {
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmDO);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == kWarpTMA) {
    // ------------------------------------------------------------ producer
    if (lane == 0 && n > 0) {
      mbar_arrive_expect_tx(kv_full, 2u * L::kTileBytes);
      for (int hh = 0; hh < L::kHalves; ++hh) {
        tma_load_4d(base + L::kOffK + hh * kHalfBytes, &tmK, kv_full, hh * 64, kvh, k0, b);
        tma_load_4d(base + L::kOffV + hh * kHalfBytes, &tmV, kv_full, hh * 64, kvh, k0, b);
      }
      bool ok = true;
      int it = 0;
      for (; it < n; ++it) {
        const int s = it % S;
        const int h = kvh * p.G + it / nqe;
        const int q0 = (qfirst + it % nqe) * kBQ;
        ok = mbar_wait(qd_empty(s), ((it / S) & 1) ^ 1, abort_flag, to);
        if (!ok) break;
        mbar_arrive_expect_tx(qd_full(s), 2u * L::kTileBytes);
        for (int hh = 0; hh < L::kHalves; ++hh) {
          tma_load_4d(base + L::kOffQ + s * L::kTileBytes + hh * kHalfBytes, &tmQ, qd_full(s), hh * 64, h, q0,
                      b);
          tma_load_4d(base + L::kOffDO + s * L::kTileBytes + hh * kHalfBytes, &tmDO, qd_full(s), hh * 64, h,
                      q0, b);
        }
      }
      if (!ok) {
        volatile int no_abort = 0;
        for (int i2 = it > S ? it - S : 0; i2 < it; ++i2)
          mbar_wait(qd_full(i2 % S), (i2 / S) & 1, &no_abort, 200000000ull);
        mbar_wait(kv_full, 0, &no_abort, 200000000ull);
      }
    }
  } else if (warp == kWarpMMA) {
    // ---------------------------------------------------------- MMA issuer
    if (lane == 0 && n > 0) {
      const uint32_t idesc_s = make_idesc_bf16(128, kBQ, 0, 0);   // K/V (A), Q/dO K-major (B)
      const uint32_t idesc_o = make_idesc_bf16(128, D, 0, 1);     // P^T/dS^T in TMEM, dO/Q MN-major
      auto issue_st = [&](int t) {          // S^T(t) = K Q(t)^T
        const uint32_t qa = base + L::kOffQ + (t % S) * L::kTileBytes;
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks)
          umma_ss(tmem + L::kTmS, desc_kmajor(base + L::kOffK, ks), desc_kmajor(qa, ks), idesc_s,
                  ks > 0 ? 1u : 0u);
      };
      auto issue_dpt = [&](int t) {         // dP^T(t) = V dO(t)^T
        const uint32_t da = base + L::kOffDO + (t % S) * L::kTileBytes;
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks)
          umma_ss(tmem + tm_dp(t), desc_kmajor(base + L::kOffV, ks), desc_kmajor(da, ks), idesc_s,
                  ks > 0 ? 1u : 0u);
      };
      // test hook: `drain` has no arrival yet
      bool ok = !p.test_stall || mbar_wait(drain, 0, abort_flag, to);
      ok = ok && mbar_wait(kv_full, 0, abort_flag, to) && mbar_wait(qd_full(0), 0, abort_flag, to);
      if (ok) {
        tc_fence_after();
        issue_st(0);
        issue_dpt(0);
        umma_commit(s_full);
      }
      for (int it = 0; ok && it < n; ++it) {
        const bool more = it + 1 < n;
        ok = mbar_wait(sd_read, it & 1, abort_flag, to);
        if (ok && more) ok = mbar_wait(qd_full((it + 1) % S), ((it + 1) / S) & 1, abort_flag, to);
        if (!ok) break;
        tc_fence_after();
        if (more) {
          issue_st(it + 1);
          if constexpr (L::kDPBufs == 2) {
            // the other buffer's P^T / dS^T (iteration it-1) were read by
            // dV / dK issued before this
            issue_dpt(it + 1);
            umma_commit(s_full);
          }
        }
        ok = mbar_wait(p_full(it & 1), (it >> 1) & 1, abort_flag, to);
        if (!ok) break;
        tc_fence_after();
        const uint32_t qa = base + L::kOffQ + (it % S) * L::kTileBytes;
        const uint32_t da = base + L::kOffDO + (it % S) * L::kTileBytes;
        const uint32_t pb = tm_dp(it);
#pragma unroll
        for (int ks = 0; ks < kBQ / 16; ++ks)       // dV += P^T dO
          umma_ts(tmem + L::kTmDV, tmem + pb + 16u + packed_col(ks), desc_mnmajor<D>(da, ks), idesc_o,
                  (it > 0 || ks > 0) ? 1u : 0u);
#pragma unroll
        for (int ks = 0; ks < kBQ / 16; ++ks)       // dK += dS^T Q
          umma_ts(tmem + L::kTmDK, tmem + pb + packed_col(ks), desc_mnmajor<D>(qa, ks), idesc_o,
                  (it > 0 || ks > 0) ? 1u : 0u);
        umma_commit(qd_empty(it % S));
        if (L::kDPBufs == 1 && more) {
          issue_dpt(it + 1);                // over P^T / dS^T(it), after dV / dK read them
          umma_commit(s_full);
        }
      }
      if (ok) umma_commit(done);
      if (!ok) {
        volatile int no_abort = 0;
        umma_commit(drain);
        mbar_wait(drain, 0, &no_abort, 200000000ull);
      }
    }
  } else {
    // ------------------------------------------------- elementwise + epilogue
    // warp w: TMEM lanes 32 (w % 4) .. +31 (key rows), query columns of group w / 4
    const int r = (warp & 3) * 32 + lane;
    const int grp = warp >> 2;
    const uint32_t lane_base = uint32_t((warp & 3) * 32) << 16;
    const int j = k0 + r;
    const bool key_ok = j < Lb;
    const uint64_t cl2 = f2_pack(p.scale_log2, p.scale_log2);
    bool aborted = false;
    // D = 64: warps 0-3 bring iteration it2's lse and Dsum rows (one query row
    // per thread) into buffer it2 & 1 with 4-byte asynchronous copies, one
    // iteration ahead, so their latency is off the critical path; rows past
    // Sq are zero.  D = 128 (twice the tensor work per iteration, which hides
    // the loads) reads them at the top of each iteration: measured on B300,
    // the copies one iteration ahead made causal_long 4 % slower there while
    // bert_base (D = 64) gained 7 %.
    constexpr bool kRowsAhead = (D == 64);
    auto fill_rows = [&](int it2) {
      const int h2 = kvh * p.G + it2 / nqe;
      const int i = (qfirst + it2 % nqe) * kBQ + r;
      float* nl = rowv + (it2 & 1) * 2 * kBQ;
      if (i < p.Sq) {
        const size_t ri = (size_t(b) * p.Hq + h2) * p.Sq + i;
        asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(nl + r)), "l"(p.lse + ri) : "memory");
        asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(nl + kBQ + r)), "l"(p.dsum + ri)
                     : "memory");
      } else {
        nl[r] = 0.f;
        nl[kBQ + r] = 0.f;
      }
      asm volatile("cp.async.commit_group;" ::: "memory");
    };
    if (kRowsAhead && grp == 0 && n > 0) fill_rows(0);
    for (int it = 0; it < n; ++it) {
      const int q0 = (qfirst + it % nqe) * kBQ;
      const int buf = it & 1;
      float* nlrow = rowv + buf * 2 * kBQ;     // -lse * log2(e) of the tile's query rows
      float* ndrow = nlrow + kBQ;              // -Dsum
      if (grp == 0) {
        if constexpr (kRowsAhead) {
          // buffer `buf` was filled one iteration ago: each thread waits for
          // its own copies and scales its row in place
          asm volatile("cp.async.wait_group 0;" ::: "memory");
          nlrow[r] = -nlrow[r] * kLog2e;
          ndrow[r] = -ndrow[r];
        } else {
          // buffer `buf` was last read two iterations ago, before every
          // warp's arrival on row_full for the previous iteration, which the
          // writers have waited for
          const int i = q0 + r;
          const size_t ri = (size_t(b) * p.Hq + kvh * p.G + it / nqe) * p.Sq + i;
          nlrow[r] = i < p.Sq ? -p.lse[ri] * kLog2e : 0.f;
          ndrow[r] = i < p.Sq ? -p.dsum[ri] : 0.f;
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(row_full(buf));
      const bool ok = __all_sync(0xffffffffu, mbar_wait(row_full(buf), (it >> 1) & 1, abort_flag, to) &&
                                                 mbar_wait(s_full, it & 1, abort_flag, to));
      if (!ok) {
        aborted = true;
        break;
      }
      tc_fence_after();
      // admissible query columns c (within this group) of this key row: lo <= c < hi
      const int qg = q0 + grp * 32;
      int lo = 0;
      const int hi = min(32, p.Sq - qg);
      if (p.causal) lo = max(0, j - diag - qg);
      if (!key_ok) lo = 32;
      const bool full = __all_sync(0xffffffffu, lo == 0 && hi == 32);
      uint32_t sv[32], dp[32], pw[16], dw[16];
      const uint32_t pcol = tm_dp(it) + uint32_t(grp) * 32u;   // this group's dP^T columns
      tmem_ld_32x32b_x32(tmem + lane_base + L::kTmS + uint32_t(grp) * 32u, sv);
      tmem_ld_32x32b_x32(tmem + lane_base + pcol, dp);
      tmem_ld_wait_x32(sv);
      tmem_ld_wait_x32(dp);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(sd_read);
      // Every warp has arrived on row_full for this iteration, so none still
      // reads the other buffer (iteration it - 1): refill it for iteration
      // it + 1, after this iteration's TMEM loads have been issued.
      if (kRowsAhead && grp == 0 && it + 1 < n) fill_rows(it + 1);
      const float* nl = nlrow + grp * 32;
      const float* nd = ndrow + grp * 32;
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const float4 l4 = *reinterpret_cast<const float4*>(nl + 4 * e);
        const float4 d4 = *reinterpret_cast<const float4*>(nd + 4 * e);
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          const int c0 = 4 * e + 2 * u;
          float x0, x1, p0, p1, t0, t1;
          f2_unpack(f2_fma(f2_pack(__uint_as_float(sv[c0]), __uint_as_float(sv[c0 + 1])), cl2,
                           u ? f2_pack(l4.z, l4.w) : f2_pack(l4.x, l4.y)),
                    x0, x1);
          p0 = ex2_approx(x0);
          p1 = ex2_approx(x1);
          if (!full) {
            p0 = (c0 >= lo && c0 < hi) ? p0 : 0.f;
            p1 = (c0 + 1 >= lo && c0 + 1 < hi) ? p1 : 0.f;
          }
          f2_unpack(f2_add(f2_pack(__uint_as_float(dp[c0]), __uint_as_float(dp[c0 + 1])),
                           u ? f2_pack(d4.z, d4.w) : f2_pack(d4.x, d4.y)),
                    t0, t1);
          pw[c0 / 2] = pack_bf16x2(p0, p1);
          dw[c0 / 2] = pack_bf16x2(p0 * t0, p1 * t1);
        }
      }
      // dS^T and P^T (bf16 pairs) over this group's own dP^T columns
      tmem_st_32x32b_x16(tmem + lane_base + pcol, dw);
      tmem_st_32x32b_x16(tmem + lane_base + pcol + 16u, pw);
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(p_full(it & 1));
    }
    if (kRowsAhead && grp == 0) asm volatile("cp.async.wait_group 0;" ::: "memory");   // no copy in flight at exit
    // epilogue: column group grp < D / 32 writes columns [32 grp, 32 grp + 32)
    // of the key row's dK and dV
    const size_t orow = ((size_t(b) * p.Sk + j) * p.Hkv + kvh) * D + size_t(grp) * 32;
    if (n == 0 && j < p.Sk && grp < D / 32) {
      store_zero_row(p.dv + orow, 32);       // no query sees these keys
      store_zero_row(p.dk + orow, 32);
    }
    if (n > 0 && !aborted) {
      const bool ok = __all_sync(0xffffffffu, mbar_wait(done, 0, abort_flag, to));
      tc_fence_after();
      if (ok && grp < D / 32) {
        uint32_t v[32];
        tmem_ld_32x32b_x32(tmem + lane_base + L::kTmDV + uint32_t(grp) * 32u, v);
        tmem_ld_wait_x32(v);
        if (j < p.Sk) store_row32(p.dv + orow, v, 1.f);
        tmem_ld_32x32b_x32(tmem + lane_base + L::kTmDK + uint32_t(grp) * 32u, v);
        tmem_ld_wait_x32(v);
        if (j < p.Sk) store_row32(p.dk + orow, v, p.scale);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kWarpMMA) {
    tc_fence_after();
    tmem_dealloc(tmem, L::kTmCols);
  }
}

}  // namespace bwd
}  // namespace gqa
