// prefill_sm103.cuh -- bf16 grouped-query attention forward (prefill) for
// sm_103a: TMA + tcgen05.mma with TMEM accumulators, warp-specialised and
// persistent.
//
// Method (sources cited by page title and section):
//  * "3个GQA核心优化技巧" (blog.gitcode.com), "GQA的分组共享机制" and
//    "Flash-Attention的稀疏分组优化": the G = Hq/Hkv query heads of a group
//    read one K/V head (kvh = h / G), and a K/V block brought on chip once is
//    reused by every query head of the group.  Here the G heads of a group
//    are packed into the M dimension of one 128-row MMA tile (row = token *
//    G + head-in-group), so each K/V tile is loaded once per CTA and feeds
//    all of them.
//  * "FlashAttention Serisi" (webturing.pages.dev), "Ana fikir": scores are
//    consumed tile by tile with a running maximum and running sum (online
//    softmax) and never written to global memory; "V3 ve donanım uyumu":
//    producer warps move data while consumer warps compute.
//
// Work unit: batch b, K/V head kvh, and 2 consecutive Q tiles of Mq =
// floor(128/G) tokens x G heads each.  The grid is persistent (at most one
// CTA per SM); CTA c starts with unit c and then claims units from a counter
// in global memory (dynamic scheduling evens out units of different length).
// Causal launches number the units longest first.  Warp roles (384 threads):
//   warps 0-3  softmax + epilogue for Q tile 0 (thread = one row = one TMEM lane)
//   warps 4-7  softmax + epilogue for Q tile 1
//   warp  8    TMA producer: the unit's Q tiles, then a K ring and a V ring
//   warp  9    MMA issuer for Q tile 0, warp 10 for Q tile 1: S_t = Q_t K^T
//              into TMEM, O_t += P_t V with P_t read from TMEM
//   warp  11   idle (it completes the third warpgroup, which hands its
//              registers to the softmax warpgroups with setmaxnreg)
// TMEM (512 columns): S0 [0,128) S1 [128,256) O0 [256,256+D) O1 [256+D,256+2D),
// and with D = 64 the unit's Q tiles Q0 [384,416) Q1 [416,448) as bf16 pairs.
//
// Schedule of Q tile t (key tiles j of a unit):
//   issuer:  QK_t(0), QK_t(1), then per j: PV_t(j), QK_t(j+2)
//   softmax: per j: P_t(j) from S_t(j) in registers; read S_t(j+1) into
//            registers; write P_t(j) (packed bf16) over S_t
// so S_t(j+1) is computed while the softmax works on tile j, and the softmax
// never waits for its own tile's matrix products in the steady state.
// QK_t(j+2) may overwrite S_t once PV_t(j) has read P_t(j): both come from the
// same issuing thread, so the tensor core runs them in that order.  One
// issuing thread per Q tile lets each thread's barrier waits overlap the
// other's MMAs.  Buffers shared by the two Q tiles (the Q set, the K/V ring
// stages) are released by both issuers.  Across units, an issuer starts the
// next unit's QK^T right after its last PV; only the first PV of a unit
// waits for the previous epilogue to have read O_t.  With D = 64 QK^T takes Q
// from TMEM: a tensor-core MMA can read about 64 bytes of shared memory per
// clock, which two shared-memory operands of a 128x128x16 step exceed by a
// factor of two, while an operand in TMEM does not count against it; the
// copy also frees the Q buffer at the start of each unit, so the next unit's
// Q lands during the current one.  Hand-offs where a whole warp takes part
// use one elected arrival per warp (fewer shared-memory atomics).
//
// Softmax details: t = s * scale * log2(e).  Each tile's row max is taken
// first, then the exponents against the reference max m, which moves only
// when the row max grows by more than 8 (log2 units), so p <= 2^8 and O_t is
// rescaled only then (after PV_t(j-1) has completed); the final division by
// l = sum p is exact for any reference.  Masked keys (j >= L_b, or
// j > i + Sk - Sq when causal) get p = 0 exactly.
#pragma once

#include "common.cuh"

namespace gqa {
namespace prefill {

constexpr int kBM = 128;       // rows per Q tile (= TMEM lanes)
constexpr int kBN = 128;       // keys per K/V tile
constexpr int kNQT = 2;        // Q tiles per work unit
constexpr int kWarpTMA = 8;
constexpr int kWarpMMA = 9;      // issues the MMAs of Q tile 0
constexpr int kWarpMMA2 = 10;    // issues the MMAs of Q tile 1
constexpr int kThreads = 384;
constexpr int kSoftmaxRegs = 224;   // 2 x 128 x 224 + 128 x 56 = 384 x 168 registers at launch
constexpr int kLaunchRegs = 168;
constexpr int kOtherRegs = 56;
constexpr float kRescaleThreshold = 8.0f;
constexpr int kUQ = 4;                // depth of the shared-memory work-unit queue
constexpr int kMaxLptB = 64;          // batch entries up to which units are claimed longest first
// consumers of a queue entry: the two MMA-issuing threads and every softmax
// warp (one elected arrival per warp)
constexpr uint32_t kUQConsumers = kNQT + kNQT * 4;

template <int D>
struct Layout {
  static constexpr int kHalves = D / 64;                    // 64-column (128-byte) halves of a row
  static constexpr int kStages = (D == 64) ? 4 : 2;         // depth of the K ring and of the V ring
  static constexpr int kQBufs = 1;                          // Q tile sets in shared memory
  // D = 64: the MMA warp copies the unit's Q tiles into TMEM (tcgen05.cp) and
  // QK^T reads A from there, which leaves the shared-memory operand bandwidth
  // to K alone; the Q buffer is free again as soon as the copies complete.
  static constexpr bool kQInTmem = (D == 64);
  static constexpr uint32_t kHalfBytes = 128u * 128u;       // 128 rows x 128 bytes
  static constexpr uint32_t kTileBytes = kHalves * kHalfBytes;
  static constexpr uint32_t kQSetBytes = kNQT * kTileBytes;
  static constexpr uint32_t kOffQ = 0;
  static constexpr uint32_t kOffK = kOffQ + kQBufs * kQSetBytes;
  static constexpr uint32_t kOffV = kOffK + kStages * kTileBytes;
  // epilogue staging: one 128-row x 64-column bf16 block (128-byte swizzle,
  // the layout of the output tensor map's box) per Q tile
  static constexpr uint32_t kOffOut = kOffV + kStages * kTileBytes;
  static constexpr uint32_t kOffBar = kOffOut + kNQT * kHalfBytes;
  // barriers: q_full[QB], q_empty[QB], k_full[S], k_empty[S], v_full[S], v_empty[S],
  //           s_full[2], p_full[2], o_done[2], o_free[2], drain, stg_free[2], stg_full[2],
  //           uq_full[kUQ], uq_empty[kUQ], s_free[2], pv_done[2], drain2
  static constexpr int kNumBars = 2 * kQBufs + 4 * kStages + 4 * kNQT + 1 + 2 * kNQT + 2 * kUQ + 2 * kNQT + 1;
  // unit queue: kUQ entries of (unit index, key length)
  static constexpr uint32_t kOffUQ = kOffBar + 8u * kNumBars;
  static constexpr uint32_t kOffTmemSlot = kOffUQ + 32u * kUQ;
  static constexpr uint32_t kOffAbort = kOffTmemSlot + 8u;
  static constexpr uint32_t kOffOrd = kOffAbort + 8u;         // [kMaxLptB] batch entries, longest first
  static constexpr uint32_t kBytes = kOffOrd + 4u * kMaxLptB;
  static constexpr uint32_t kSmemAlloc = kBytes + 1024u;    // slack to align the base to 1024 B
  // V is the MN-major B operand: 8-key groups 1024 B apart (SBO); the second
  // 64-wide head-dim half (D = 128) is kHalfBytes further (LBO).  With D = 64
  // the LBO is never used and is set to 1024 so the descriptor stays inside
  // the stage whichever way the two offsets are read.
  static constexpr uint32_t kVLbo = (D == 64) ? 1024u : kHalfBytes;
  static constexpr uint32_t kTmCols = 512;
  static constexpr uint32_t kTmS0 = 0, kTmS1 = 128;
  static constexpr uint32_t kTmO0 = 256, kTmO1 = 256 + D;
  static constexpr uint32_t kTmQ0 = 256 + 2 * D, kTmQ1 = 256 + 2 * D + D / 2;   // D = 64 only: bf16 pairs
  static_assert(!kQInTmem || kTmQ1 + D / 2 <= kTmCols, "TMEM column map overflows");
};

struct Params {
  __nv_bfloat16* out;     // [B, Sq, Hq, D]; packed: [total_q, Hq, D]
  float* lse;             // [B, Hq, Sq]; packed: [Hq, total_q]; or nullptr
  const int* seqlens;     // [B] or nullptr (dense layout only)
  // Packed (variable-length) layout when cu_q != nullptr: sequence b owns
  // query rows [cu_q[b], cu_q[b+1]) and key rows [cu_k[b], cu_k[b+1]); the
  // tensor maps then see one batch entry of total_q / total_k rows, and Sq /
  // Sk are the largest sequence lengths.
  const int* cu_q;
  const int* cu_k;
  int total_q, total_k;
  int lse_stride;         // Sq (dense) or total_q (packed)
  // Block sparsity (dense layout): bmask [n_qb, n_kb] uint8, nonzero = query
  // block i // bs may attend to key block j // bs; bs = 64 or 128 and
  // Sk <= 8192 (one 64-bit word of 128-key tiles per unit).
  const uint8_t* bmask;
  int bs, n_qb, n_kb;
  int B, Hq, Hkv, G, Sq, Sk;
  int Mq;                 // tokens per Q tile (G * Mq <= 128)
  int n_qblk;             // ceil(Sq / (kNQT * Mq))
  int n_units;            // n_qblk * B * Hkv
  // Work-unit scheduler of this launch: sched[0] counts units claimed past
  // the first gridDim.x, sched[1] counts CTAs that finished; the last CTA to
  // finish sets both back to zero for the next launch that uses the slot.
  unsigned int* sched;
  int causal;
  float scale_log2;       // scale * log2(e)
  unsigned long long timeout_ns;
  // Test hook: when nonzero, Q tile 0's MMA issuer first waits on a barrier
  // that nothing arrives on, so the wait runs out after timeout_ns and the
  // whole CTA takes its abort path (device timeout status, drained copies
  // and MMAs, TMEM freed).
  int test_stall;
};

struct Unit {
  int b, kvh, q0, Lb, n_tiles;
  int Lq;                  // query rows of the sequence (Sq when dense)
  int qbase, kbase;        // first packed row of the sequence (0 when dense)
  int tb;                  // batch coordinate of the tensor maps (b, or 0 when packed)
  int diag;                // causal: query row i sees keys j <= i + diag
  bool has_rows;           // the unit holds at least one query row
  uint64_t act;            // block sparsity: active 128-key tiles (n_tiles = their count)
  bool bad_len;
};

// Lengths and packed row offsets of a work unit's sequence, read by the TMA
// warp one unit ahead and passed on through the unit queue.
struct SeqInfo {
  int Lk, Lq, qbase, kbase;
  uint32_t act_lo, act_hi;   // block sparsity: the unit's active 128-key tiles
};

// One bit per byte of w: bit e set when byte e is nonzero.
DEVI uint32_t nonzero_bytes4(uint32_t w) {
  uint32_t t = w | (w >> 4);
  t |= t >> 2;
  t |= t >> 1;
  return (t & 1u) | ((t >> 7) & 2u) | ((t >> 14) & 4u) | ((t >> 21) & 8u);
}

// Bits of row qb of the block mask: bit kb set when block (qb, kb) is kept.
// Whole 16-byte chunks of the row by vector loads when the row is 16-byte
// aligned, the rest byte by byte; nothing past the row is read.
DEVI void mask_row_bits(const Params& p, int qb, uint64_t& lo, uint64_t& hi) {
  lo = 0;
  hi = 0;
  const uint8_t* row = p.bmask + size_t(qb) * p.n_kb;
  int kb = 0;
  if ((reinterpret_cast<uintptr_t>(row) & 15u) == 0) {
    for (; kb + 16 <= p.n_kb; kb += 16) {
      uint4 w;
      asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];"
                   : "=r"(w.x), "=r"(w.y), "=r"(w.z), "=r"(w.w)
                   : "l"(row + kb));
      const uint64_t bits = uint64_t(nonzero_bytes4(w.x)) | (uint64_t(nonzero_bytes4(w.y)) << 4) |
                            (uint64_t(nonzero_bytes4(w.z)) << 8) | (uint64_t(nonzero_bytes4(w.w)) << 12);
      if (kb < 64) lo |= bits << kb; else hi |= bits << (kb - 64);
    }
  }
  for (; kb < p.n_kb; ++kb) {
    const uint64_t bit = row[kb] ? 1ull : 0ull;
    if (kb < 64) lo |= bit << kb; else hi |= bit << (kb - 64);
  }
}

// The 32 bits of x at even positions, packed (bit 2k -> bit k).
DEVI uint64_t even_bits(uint64_t x) {
  x &= 0x5555555555555555ull;
  x = (x | (x >> 1)) & 0x3333333333333333ull;
  x = (x | (x >> 2)) & 0x0F0F0F0F0F0F0F0Full;
  x = (x | (x >> 4)) & 0x00FF00FF00FF00FFull;
  x = (x | (x >> 8)) & 0x0000FFFF0000FFFFull;
  x = (x | (x >> 16)) & 0x00000000FFFFFFFFull;
  return x;
}

// Key-block bits (lo: blocks 0-63, hi: 64-127) -> 128-key-tile bits.  With
// bs = 128 a tile is one block; with bs = 64 tile j holds blocks 2j (`half`
// 0) and 2j+1 (`half` 1).
DEVI uint64_t tiles_of_blocks(int bs, uint64_t lo, uint64_t hi, int half) {
  if (bs == 128) return lo;
  const uint64_t a = half ? lo >> 1 : lo, b = half ? hi >> 1 : hi;
  return even_bits(a) | (even_bits(b) << 32);
}

// Position of work unit u.  Non-causal: u = qidx * (B * Hkv) + b * Hkv + kvh,
// so the units running at one time spread over every (b, kvh) and their
// lengths even out.  Causal: u = (b * Hkv + kvh) * n_qblk + qidx, so the
// units running at one time are Q blocks of the same one or two (b, kvh):
// they read the same K/V tiles, which then come from L2 instead of DRAM
// (a long causal launch holds far more K/V than L2 does); qidx counts the
// Q blocks longest first (unit_info), which keeps the tail short.
struct UnitPos {
  int u, qidx, b, kvh;
};
DEVI UnitPos upos_of(const Params& p, int u) {
  UnitPos x;
  x.u = u;
  int bh;
  if (p.causal) {
    bh = u / p.n_qblk;
    x.qidx = u - bh * p.n_qblk;
  } else {
    const int bh_count = p.B * p.Hkv;
    x.qidx = u / bh_count;
    bh = u - x.qidx * bh_count;
  }
  x.b = bh / p.Hkv;
  x.kvh = bh - x.b * p.Hkv;
  return x;
}

// Key length of the unit's batch entry.
DEVI int ldg_nc_i32(const int* a) {
  int v;
  asm volatile("ld.global.nc.b32 %0, [%1];" : "=r"(v) : "l"(a));
  return v;
}
template <bool kPacked>
DEVI SeqInfo unit_seq(const Params& p, const UnitPos& x) {
  SeqInfo q;
  if constexpr (kPacked) {
    const int q0 = ldg_nc_i32(p.cu_q + x.b), q1 = ldg_nc_i32(p.cu_q + x.b + 1);
    const int k0 = ldg_nc_i32(p.cu_k + x.b), k1 = ldg_nc_i32(p.cu_k + x.b + 1);
    q.Lq = q1 - q0;
    q.Lk = k1 - k0;
    q.qbase = q0;
    q.kbase = k0;
  } else {
    q.Lk = p.seqlens ? ldg_nc_i32(p.seqlens + x.b) : p.Sk;
    q.Lq = p.Sq;
    q.qbase = 0;
    q.kbase = 0;
  }
  return q;
}

// Claims the next work unit of this launch (returns gridDim.x + a running
// count).  Volatile so that it is issued where it is written, one unit ahead
// of its use.
DEVI int claim_unit(const Params& p) {
  unsigned int v;
  asm volatile("atom.global.add.u32 %0, [%1], 1;" : "=r"(v) : "l"(p.sched) : "memory");
  return int(gridDim.x + v);
}

// Work unit -> (b, kvh, first token, key length, number of key tiles); len is
// unit_len of the same unit.
template <bool kPacked, bool kSparse>
DEVI Unit unit_info(const Params& p, const UnitPos& x, const SeqInfo& sq) {
  Unit U;
  const int qblk = p.causal ? p.n_qblk - 1 - x.qidx : x.qidx;   // causal: longest units first
  U.b = x.b;
  U.kvh = x.kvh;
  U.q0 = qblk * kNQT * p.Mq;
  int Lb = sq.Lk, Lq = kPacked ? sq.Lq : p.Sq;
  U.bad_len = (Lb < 0 || Lb > p.Sk || Lq < 0 || Lq > p.Sq);
  if (kPacked)
    U.bad_len = U.bad_len || sq.qbase < 0 || sq.kbase < 0 || sq.qbase > p.total_q - Lq ||
                sq.kbase > p.total_k - Lb;
  if (U.bad_len) {
    // a dense unit still writes zeros for its rows; a packed one cannot
    // place its rows and writes nothing
    Lb = 0;
    if (kPacked) Lq = 0;
  }
  U.Lb = Lb;
  U.Lq = Lq;
  U.qbase = kPacked ? sq.qbase : 0;
  U.kbase = kPacked ? sq.kbase : 0;
  U.tb = kPacked ? 0 : x.b;
  U.has_rows = U.q0 < Lq;
  // bottom-right aligned diagonal: of the padded sizes (dense) or of the
  // sequence's own lengths (packed)
  U.diag = kPacked ? Lb - Lq : p.Sk - p.Sq;
  const int q_last = min(U.q0 + kNQT * p.Mq, Lq) - 1;
  int kmax = Lb;
  if (p.causal) kmax = min(kmax, q_last + U.diag + 1);
  U.n_tiles = (U.has_rows && kmax > 0) ? (kmax + kBN - 1) / kBN : 0;
  if constexpr (kSparse) {
    // the tiles within reach (n_tiles <= 64: Sk <= 8192) that a block of the
    // unit's rows keeps; n_tiles becomes their count
    const uint64_t reach = U.n_tiles >= 64 ? ~0ull : ((1ull << U.n_tiles) - 1);
    U.act = ((uint64_t(sq.act_hi) << 32) | sq.act_lo) & reach;
    U.n_tiles = __popcll(U.act);
  }
  return U;
}

// Block sparsity: the 128-key tiles that any query block of the unit keeps
// (U is the unit's dense geometry).
DEVI uint64_t unit_active_tiles(const Params& p, const Unit& U) {
  if (!U.has_rows || U.n_tiles == 0) return 0;
  const int q_last = min(U.q0 + kNQT * p.Mq, U.Lq) - 1;
  uint64_t act = 0;
  for (int qb = U.q0 / p.bs; qb <= q_last / p.bs; ++qb) {
    uint64_t lo, hi;
    mask_row_bits(p, qb, lo, hi);
    act |= tiles_of_blocks(p.bs, lo, hi, 0) | tiles_of_blocks(p.bs, lo, hi, 1);
  }
  return act;
}

template <int D, bool kPacked, bool kSparse>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                   const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO,
                   const Params p) {
  using L = Layout<D>;
  constexpr int S = L::kStages;
  constexpr int QB = L::kQBufs;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  const uint32_t base = (raw_addr + 1023u) & ~1023u;
  uint8_t* sbase = smem_raw + (base - raw_addr);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int rows_per_tile = p.G * p.Mq;

  auto bar = [&](int i) -> uint32_t { return base + L::kOffBar + 8u * uint32_t(i); };
  auto q_full = [&](int i) { return bar(i); };
  auto q_empty = [&](int i) { return bar(QB + i); };
  auto k_full = [&](int s) { return bar(2 * QB + s); };
  auto k_empty = [&](int s) { return bar(2 * QB + S + s); };
  auto v_full = [&](int s) { return bar(2 * QB + 2 * S + s); };
  auto v_empty = [&](int s) { return bar(2 * QB + 3 * S + s); };
  auto s_full = [&](int t) { return bar(2 * QB + 4 * S + t); };
  auto p_full = [&](int t) { return bar(2 * QB + 4 * S + kNQT + t); };
  auto o_done = [&](int t) { return bar(2 * QB + 4 * S + 2 * kNQT + t); };
  auto o_free = [&](int t) { return bar(2 * QB + 4 * S + 3 * kNQT + t); };
  const uint32_t drain = bar(2 * QB + 4 * S + 4 * kNQT);
  auto stg_free = [&](int t) { return bar(2 * QB + 4 * S + 4 * kNQT + 1 + t); };
  auto stg_full = [&](int t) { return bar(2 * QB + 4 * S + 5 * kNQT + 1 + t); };
  auto uq_full = [&](int i) { return bar(2 * QB + 4 * S + 6 * kNQT + 1 + i); };
  auto uq_empty = [&](int i) { return bar(2 * QB + 4 * S + 6 * kNQT + 1 + kUQ + i); };
  auto s_free = [&](int t) { return bar(2 * QB + 4 * S + 6 * kNQT + 1 + 2 * kUQ + t); };
  auto pv_done = [&](int t) { return bar(2 * QB + 4 * S + 7 * kNQT + 1 + 2 * kUQ + t); };
  const uint32_t drain2 = bar(2 * QB + 4 * S + 8 * kNQT + 1 + 2 * kUQ);

  volatile int* abort_flag = reinterpret_cast<volatile int*>(sbase + L::kOffAbort);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sbase + L::kOffTmemSlot);
  const uint64_t to = p.timeout_ns;
  // [kUQ][8]: unit, then the SeqInfo fields Lk, Lq, qbase, kbase
  volatile int* uq = reinterpret_cast<volatile int*>(sbase + L::kOffUQ);
  // Consumer side of the unit queue: entry k's (unit, key length), or
  // n_units when the wait gave up.  A whole warp (softmax) releases the
  // entry with one arrival once every lane has read it; a single thread
  // (MMA issuer) arrives itself.
  auto next_unit = [&](uint32_t k, SeqInfo& sq, bool& ok, bool whole_warp) -> int {
    const int i = int(k % kUQ);
    ok = mbar_wait(uq_full(i), (k / kUQ) & 1, abort_flag, p.timeout_ns);
    int u = p.n_units;
    if (ok) {
      u = uq[8 * i];
      sq.Lk = uq[8 * i + 1];
      if constexpr (kPacked) {
        sq.Lq = uq[8 * i + 2];
        sq.qbase = uq[8 * i + 3];
        sq.kbase = uq[8 * i + 4];
      }
      if constexpr (kSparse) {
        sq.act_lo = uint32_t(uq[8 * i + 5]);
        sq.act_hi = uint32_t(uq[8 * i + 6]);
      }
    }
    if (whole_warp) {
      __syncwarp();
      if (lane == 0) mbar_arrive(uq_empty(i));
    } else {
      mbar_arrive(uq_empty(i));
    }
    return u;
  };

  if (threadIdx.x == 0) {
    // buffers shared by the Q tiles are released by both MMA-issuing threads
    for (int i = 0; i < QB; ++i) {
      mbar_init(q_full(i), 1);
      mbar_init(q_empty(i), kNQT);
    }
    for (int s = 0; s < S; ++s) {
      mbar_init(k_full(s), 1);
      mbar_init(k_empty(s), kNQT);
      mbar_init(v_full(s), 1);
      mbar_init(v_empty(s), kNQT);
    }
    for (int t = 0; t < kNQT; ++t) {
      mbar_init(s_full(t), 1);
      mbar_init(p_full(t), 4);         // one arrival per softmax warp of the tile
      mbar_init(s_free(t), 4);
      mbar_init(pv_done(t), 1);
      mbar_init(o_done(t), 1);
      mbar_init(o_free(t), 4);
      mbar_init(stg_free(t), 1);
      mbar_init(stg_full(t), 4);
    }
    for (int i = 0; i < kUQ; ++i) {
      mbar_init(uq_full(i), 1);
      mbar_init(uq_empty(i), kUQConsumers);
    }
    mbar_init(drain, 1);
    mbar_init(drain2, 1);
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
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
    tma_prefetch_desc(&tmO);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp >= 8) {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kOtherRegs));
  if (warp == kWarpTMA) {
    // ------------------------------------------------------------ producer
    // Non-causal launches whose entries have their own key lengths (dense
    // with seqlens, or packed) and B <= kMaxLptB hand out units longest
    // first: batch entries in order of decreasing key length (ties by index),
    // all units of an entry together, so the units left at the end of the
    // launch are the shortest and the last SMs to finish wait least.  The warp
    // ranks the B lengths: lane b counts the entries that sort before entry b.
    int* ord = reinterpret_cast<int*>(sbase + L::kOffOrd);
    const bool lpt = !kSparse && !p.causal && (kPacked || p.seqlens != nullptr) && p.B <= kMaxLptB;
    auto key_len_of = [&](int bb) -> int {
      if constexpr (kPacked) return ldg_nc_i32(p.cu_k + bb + 1) - ldg_nc_i32(p.cu_k + bb);
      return ldg_nc_i32(p.seqlens + bb);
    };
    if (lpt) {
      const int L0 = lane < p.B ? key_len_of(lane) : 0;
      const int L1 = lane + 32 < p.B ? key_len_of(lane + 32) : 0;
      int r0 = 0, r1 = 0;
      for (int b2 = 0; b2 < p.B; ++b2) {
        const int Lx = __shfl_sync(0xffffffffu, b2 < 32 ? L0 : L1, b2 & 31);
        r0 += (Lx > L0 || (Lx == L0 && b2 < lane)) ? 1 : 0;
        r1 += (Lx > L1 || (Lx == L1 && b2 < lane + 32)) ? 1 : 0;
      }
      if (lane < p.B) ord[r0] = lane;
      if (lane + 32 < p.B) ord[r1] = lane + 32;
      __syncwarp();
    }
    // claim index c -> unit index (the identity unless longest first)
    auto unit_of = [&](int c) -> int {
      if (!lpt || c >= p.n_units) return c;
      const int per_b = p.n_qblk * p.Hkv;
      const int bi = c / per_b, rem = c - bi * per_b;
      const int qidx = rem / p.Hkv, kvh = rem - qidx * p.Hkv;
      return qidx * (p.B * p.Hkv) + ord[bi] * p.Hkv + kvh;
    };
    if (lane == 0) {
      uint32_t kv_it = 0;       // K/V tiles issued so far (ring position)
      uint32_t qn = 0;          // units with work so far (Q buffer position)
      bool ok = true;
      bool k_only = false;
      const uint32_t q_bytes = uint32_t(kNQT * L::kHalves * 64 * 2 * rows_per_tile);
      // Work units are claimed at run time (the first claim index is
      // blockIdx.x; the grid never exceeds the unit count), one unit ahead,
      // mapped to a unit by unit_of and published to the MMA and softmax
      // warps through the unit queue; a unit index past the last unit ends
      // every role's loop.
      int u_next = unit_of(int(blockIdx.x));
      for (uint32_t k = 0; ok; ++k) {
        const int u = u_next;
        const int i = int(k % kUQ);
        ok = mbar_wait(uq_empty(i), ((k / kUQ) & 1) ^ 1, abort_flag, to);
        if (!ok) break;
        const UnitPos x = upos_of(p, u < p.n_units ? u : 0);
        SeqInfo sq{0, 0, 0, 0};
        if (u < p.n_units) sq = unit_seq<kPacked>(p, x);
        if constexpr (kSparse) {
          if (u < p.n_units) {
            const uint64_t act = unit_active_tiles(p, unit_info<kPacked, false>(p, x, sq));
            sq.act_lo = uint32_t(act);
            sq.act_hi = uint32_t(act >> 32);
          }
        }
        if (u < p.n_units) u_next = unit_of(claim_unit(p));
        uq[8 * i] = u;
        uq[8 * i + 1] = sq.Lk;
        uq[8 * i + 2] = sq.Lq;
        uq[8 * i + 3] = sq.qbase;
        uq[8 * i + 4] = sq.kbase;
        if constexpr (kSparse) {
          uq[8 * i + 5] = int(sq.act_lo);
          uq[8 * i + 6] = int(sq.act_hi);
        }
        mbar_arrive(uq_full(i));        // release: the entry is visible to the consumers
        if (u >= p.n_units) break;
        const Unit U = unit_info<kPacked, kSparse>(p, x, sq);
        if (U.bad_len) raise_error(kErrBounds);
        if (U.n_tiles == 0) continue;
        const int qb = int(qn % QB);
        ok = mbar_wait(q_empty(qb), ((qn / QB) & 1) ^ 1, abort_flag, to);
        if (!ok) break;
        mbar_arrive_expect_tx(q_full(qb), q_bytes);
        for (int t = 0; t < kNQT; ++t)
          for (int h = 0; h < L::kHalves; ++h)
            tma_load_4d(base + L::kOffQ + qb * L::kQSetBytes + t * L::kTileBytes + h * L::kHalfBytes, &tmQ,
                        q_full(qb), h * 64, U.kvh * p.G, U.qbase + U.q0 + t * p.Mq, U.tb);
        ++qn;
        uint64_t act_rem = kSparse ? U.act : 0ull;     // block sparsity: active tiles still to load
        for (int j = 0; j < U.n_tiles; ++j) {
          int tj = j;                  // key tile index (the j-th active tile when sparse)
          if constexpr (kSparse) {
            tj = __ffsll((long long)act_rem) - 1;
            act_rem &= act_rem - 1;
          }
          const int s = int(kv_it % S);
          const uint32_t ph = (kv_it / S) & 1;
          ok = mbar_wait(k_empty(s), ph ^ 1, abort_flag, to);
          if (!ok) break;
          mbar_arrive_expect_tx(k_full(s), L::kTileBytes);
          for (int h = 0; h < L::kHalves; ++h)
            tma_load_4d(base + L::kOffK + s * L::kTileBytes + h * L::kHalfBytes, &tmK, k_full(s), h * 64,
                        U.kvh, U.kbase + tj * kBN, U.tb);
          ok = mbar_wait(v_empty(s), ph ^ 1, abort_flag, to);
          if (!ok) {
            k_only = true;     // K of ring position kv_it is in flight, V is not
            break;
          }
          mbar_arrive_expect_tx(v_full(s), L::kTileBytes);
          for (int h = 0; h < L::kHalves; ++h)
            tma_load_4d(base + L::kOffV + s * L::kTileBytes + h * L::kHalfBytes, &tmV, v_full(s), h * 64,
                        U.kvh, U.kbase + tj * kBN, U.tb);
          ++kv_it;
        }
      }
      if (!ok) {
        // aborted: let the copies already in flight land before the CTA exits.
        // Each waited phase belongs to the last load issued into its buffer,
        // so it completes (or has completed) exactly once.
        volatile int no_abort = 0;
        const uint32_t first = kv_it > uint32_t(S) ? kv_it - S : 0u;
        for (uint32_t it = first; it < kv_it; ++it) {
          mbar_wait(k_full(int(it % S)), (it / S) & 1, &no_abort, 200000000ull);
          mbar_wait(v_full(int(it % S)), (it / S) & 1, &no_abort, 200000000ull);
        }
        if (k_only) mbar_wait(k_full(int(kv_it % S)), (kv_it / S) & 1, &no_abort, 200000000ull);
        if (qn > 0) mbar_wait(q_full(int((qn - 1) % QB)), ((qn - 1) / QB) & 1, &no_abort, 200000000ull);
      }
    }
  } else if (warp == kWarpMMA || warp == kWarpMMA2) {
    // --------------------------------------------------------- MMA issuers
    // One thread per Q tile t issues that tile's MMAs in the order
    //   QK_t(0), QK_t(1), then per key tile j: PV_t(j), QK_t(j+2).
    // P_t(j) is written over S_t once the softmax has read S_t(j+1) into
    // registers, so S_t(j+1) is computed while the softmax works on tile j,
    // and QK_t(j+2) may overwrite S_t as soon as PV_t(j) has read P_t(j)
    // (same thread, so in order).  The two threads' barrier waits overlap
    // each other's MMAs.
    if (lane == 0) {
      const int tq = warp - kWarpMMA;
      const uint32_t idesc_s = make_idesc_bf16(128, kBN, 0, 0);   // Q, K both K-major
      const uint32_t idesc_o = make_idesc_bf16(128, D, 0, 1);     // P (TMEM), V MN-major
      auto issue_s = [&](int t, int qb, int s) {
        const uint32_t qa = base + L::kOffQ + qb * L::kQSetBytes + t * L::kTileBytes;
        const uint32_t ka = base + L::kOffK + s * L::kTileBytes;
        const uint32_t dst = tmem + (t ? L::kTmS1 : L::kTmS0);
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          const uint32_t off = uint32_t(ks / 4) * L::kHalfBytes + uint32_t(ks % 4) * 32u;
          if constexpr (L::kQInTmem)
            umma_ts(dst, tmem + (t ? L::kTmQ1 : L::kTmQ0) + uint32_t(ks) * 8u, make_sdesc_sw128(ka + off, 16, 1024),
                    idesc_s, ks > 0 ? 1u : 0u);
          else
            umma_ss(dst, make_sdesc_sw128(qa + off, 16, 1024), make_sdesc_sw128(ka + off, 16, 1024),
                    idesc_s, ks > 0 ? 1u : 0u);
        }
      };
      // D = 64: the unit's Q tiles from shared memory into TMEM (executes
      // after every MMA issued before it, so the previous unit's QK^T are done)
      auto copy_q = [&](int qb, int t) {
        const uint32_t qa = base + L::kOffQ + qb * L::kQSetBytes + t * L::kTileBytes;
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks)
          tmem_cp_128x256b(tmem + (t ? L::kTmQ1 : L::kTmQ0) + uint32_t(ks) * 8u,
                           make_sdesc_sw128(qa + uint32_t(ks) * 32u, 16, 1024));
      };
      auto issue_pv = [&](int t, int s, bool acc) {
        const uint32_t va = base + L::kOffV + s * L::kTileBytes;
        const uint32_t dst = tmem + (t ? L::kTmO1 : L::kTmO0);
        const uint32_t pa = tmem + (t ? L::kTmS1 : L::kTmS0);
#pragma unroll
        for (int ks = 0; ks < kBN / 16; ++ks) {
          umma_ts(dst, pa + uint32_t(ks) * 8u, make_sdesc_sw128(va + uint32_t(ks) * 2048u, L::kVLbo, 1024),
                  idesc_o, (acc || ks > 0) ? 1u : 0u);
        }
      };
      uint32_t g = 0;           // key tiles of earlier units (K/V ring position; s_full / p_full phases)
      uint32_t qn = 0;          // units with work so far
      uint32_t n2 = 0;          // units with two or more key tiles so far (s_free / pv_done phases)
      // test hook: `drain` (tile 0's abort barrier) has no arrival yet
      bool ok = !(p.test_stall && tq == 0) || mbar_wait(drain, 0, abort_flag, to);
      for (uint32_t k = 0; ok; ++k) {
        SeqInfo sq;
        const int u = next_unit(k, sq, ok, false);
        if (!ok || u >= p.n_units) break;
        const Unit U = unit_info<kPacked, kSparse>(p, upos_of(p, u), sq);
        const int n = U.n_tiles;
        if (n == 0) continue;
        const int qb = int(qn % QB);
        // QK^T_t of the unit's key tile jj (jj = 0, 1), K from ring stage (g + jj) % S
        auto qk = [&](int jj) -> bool {
          const uint32_t it = g + uint32_t(jj);
          const int s = int(it % S);
          if (!mbar_wait(k_full(s), (it / S) & 1, abort_flag, to)) return false;
          tc_fence_after();
          issue_s(tq, qb, s);
          umma_commit(s_full(tq));
          umma_commit(k_empty(s));
          if (!L::kQInTmem && jj == n - 1) umma_commit(q_empty(qb));   // the unit's last read of Q
          return true;
        };
        ok = mbar_wait(q_full(qb), (qn / QB) & 1, abort_flag, to);
        if (!ok) break;
        tc_fence_after();
        if constexpr (L::kQInTmem) {
          copy_q(qb, tq);
          umma_commit(q_empty(qb));     // this Q tile's part of the buffer is free once copied
        }
        ok = qk(0);
        // S_t(1) may overwrite S_t(0) once the softmax has read it
        if (ok && n >= 2) ok = mbar_wait(s_free(tq), n2 & 1, abort_flag, to) && qk(1);
        for (int j = 0; ok && j < n; ++j) {
          const uint32_t it = g + uint32_t(j);
          const int s = int(it % S);
          // With a ring of four or more stages K of tile j+2 was loaded long
          // ago, so its wait goes first and hides under the P wait; with two
          // stages it shares K(j)'s stage and is loaded just in time, so it is
          // waited for after PV(j).
          constexpr bool kEarlyK = S >= 4;
          const bool more = j + 2 < n;
          const uint32_t it2 = it + 2u;
          const int s2 = int(it2 % S);
          if (kEarlyK && more) ok = mbar_wait(k_full(s2), (it2 / S) & 1, abort_flag, to);
          ok = ok && mbar_wait(v_full(s), (it / S) & 1, abort_flag, to) && mbar_wait(p_full(tq), it & 1, abort_flag, to);
          // the unit's first PV overwrites O_t: the previous epilogue must have read it
          if (ok && j == 0 && qn > 0) ok = mbar_wait(o_free(tq), (qn - 1) & 1, abort_flag, to);
          if (!ok) break;
          tc_fence_after();
          issue_pv(tq, s, j > 0);
          // Deep ring: QK_t(j+2) straight after PV_t(j), the release commits
          // after it.  Two-stage ring: V(j) is released at once (the next V
          // load waits for it) and K(j+2) is waited for here.
          if constexpr (!kEarlyK) {
            if (j == n - 2) umma_commit(pv_done(tq));   // lets the softmax rescale O_t before the last PV
            if (j == n - 1) umma_commit(o_done(tq));
            umma_commit(v_empty(s));
            if (more) {
              ok = mbar_wait(k_full(s2), (it2 / S) & 1, abort_flag, to);
              if (!ok) break;
              tc_fence_after();
            }
          }
          if (more) {
            // QK_t(j+2) follows PV_t(j) in the tensor core (same issuing thread)
            issue_s(tq, qb, s2);
            umma_commit(s_full(tq));
          }
          if constexpr (kEarlyK) {
            if (j == n - 2) umma_commit(pv_done(tq));
            if (j == n - 1) umma_commit(o_done(tq));
            umma_commit(v_empty(s));
          }
          if (more) {
            umma_commit(k_empty(s2));
            if (!L::kQInTmem && j + 3 == n) umma_commit(q_empty(qb));   // the unit's last read of Q
          }
        }
        if (n >= 2) ++n2;
        g += uint32_t(n);
        ++qn;
      }
      if (!ok) {
        // aborted: wait for the tensor core to finish what this thread issued
        volatile int no_abort = 0;
        const uint32_t db = tq ? drain2 : drain;
        umma_commit(db);
        mbar_wait(db, 0, &no_abort, 200000000ull);
      }
    }
  }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kSoftmaxRegs));
    // ------------------------------------------------------------- softmax
    const int t = warp >> 2;
    const int wq = warp & 3;
    const int r = wq * 32 + lane;
    const uint32_t lane_base = uint32_t(wq * 32) << 16;
    const uint32_t tS = tmem + lane_base + (t ? L::kTmS1 : L::kTmS0);
    const uint32_t tO = tmem + lane_base + (t ? L::kTmO1 : L::kTmO0);
    const int g = r % p.G;
    const float c = p.scale_log2;
    const uint64_t c2 = f2_pack(c, c);
    uint32_t g_tile = 0;
    uint32_t qn = 0;
    uint32_t n2 = 0;          // units with two or more key tiles so far
    uint32_t n_stage = 0;     // uses of this tile's staging block so far
    bool aborted = false;

    const int r_tok = r / p.G;   // token of this row within the Q tile
    // The next unit's queue entry is read one unit ahead, while the current
    // unit's last PV runs (before its epilogue can read O).
    SeqInfo sq_next;
    bool next_ok;
    int u_next = next_unit(0, sq_next, next_ok, true);
    next_ok = __all_sync(0xffffffffu, next_ok);
    for (uint32_t k = 0; !aborted; ++k) {
      if (!next_ok) {
        aborted = true;
        break;
      }
      if (u_next >= p.n_units) break;
      const Unit U = unit_info<kPacked, kSparse>(p, upos_of(p, u_next), sq_next);
      const int token = U.q0 + t * p.Mq + r_tok;
      const bool row_ok = (r < rows_per_tile) && (token < U.Lq);
      int limit = 0;
      if (row_ok) {
        limit = U.Lb;
        if (p.causal) limit = min(limit, token + U.diag + 1);
        limit = max(limit, 0);
      }
      float m = -INFINITY;
      float l = 0.f;

      const int n = U.n_tiles;
      // block sparsity: the unit's active tiles still to process, and the
      // tiles this row's query block keeps for its low / high 64 keys
      uint64_t act_rem = kSparse ? U.act : 0ull, row_lo = ~0ull, row_hi = ~0ull;
      if constexpr (kSparse) {
        if (row_ok) {
          uint64_t blo, bhi;
          mask_row_bits(p, token / p.bs, blo, bhi);
          row_lo = tiles_of_blocks(p.bs, blo, bhi, 0);
          row_hi = tiles_of_blocks(p.bs, blo, bhi, 1);
        }
      }
      uint32_t sv[kBN];        // S_t of the current key tile, in registers
      if (n > 0) {
        // S_t(0), read before the loop so that every tile's S is visibly
        // defined on entry (S_t(j+1) is read at the end of tile j)
        // (loaded even after a failed wait, whose tile is then skipped)
        const bool ok = mbar_wait(s_full(t), g_tile & 1, abort_flag, to);
        if (!__all_sync(0xffffffffu, ok)) aborted = true;
        tc_fence_after();
        tmem_ld_32x32b_x32(tS + 0, sv + 0);
        tmem_ld_32x32b_x32(tS + 32, sv + 32);
        tmem_ld_32x32b_x32(tS + 64, sv + 64);
        tmem_ld_32x32b_x32(tS + 96, sv + 96);
        tmem_ld_wait_x128(sv);
        if (n >= 2 && !aborted) {
          // S_t(0) is in registers: QK_t(1) may overwrite it
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(s_free(t));
        }
      } else {
#pragma unroll
        for (int i = 0; i < kBN; ++i) sv[i] = 0u;
      }
      for (int j = 0; j < n && !aborted; ++j) {
        const uint32_t gi = g_tile + uint32_t(j);
        uint32_t pall[kBN / 2];  // P_t(j) as bf16 pairs, written to TMEM at the end of the tile
        // Before P_t(j) can go over S_t: S_t(j+1) must be complete (it is
        // then read into registers), or for the unit's last tile PV_t(j-1).
        // Either way PV_t(j-1) has completed (QK_t(j+1) was issued after
        // it), which also allows rescaling O_t.
        bool waited = false;
        auto wait_next = [&]() -> bool {
          if (waited) return true;
          waited = true;
          bool okn = true;
          if (j + 1 < n)
            okn = mbar_wait(s_full(t), (gi + 1) & 1, abort_flag, to);
          else if (n >= 2)
            okn = mbar_wait(pv_done(t), n2 & 1, abort_flag, to);
          okn = __all_sync(0xffffffffu, okn);
          tc_fence_after();
          return okn;
        };

        int tj = j;             // key tile index (the j-th active tile when sparse)
        if constexpr (kSparse) {
          tj = __ffsll((long long)act_rem) - 1;
          act_rem &= act_rem - 1;
        }
        const int lim = limit - tj * kBN;
        bool ok_lo = true, ok_hi = true;   // this row keeps the tile's low / high 64 keys
        if constexpr (kSparse) {
          ok_lo = (row_lo >> tj) & 1ull;
          ok_hi = (row_hi >> tj) & 1ull;
        }
        // Keys at or past the row's limit get exactly zero weight.  When every
        // row of the warp admits every key of the tile (rows that hold no
        // query are never stored and do not count) and the scale is positive,
        // no mask is needed and the max is taken on the raw scores.  Every
        // branch below is warp-uniform.
        const bool full = __all_sync(0xffffffffu, (lim >= kBN && ok_lo && ok_hi) || !row_ok) && (c > 0.f);
        float mt = -INFINITY;
        if (full) {
#pragma unroll
          for (int i = 0; i < kBN; i += 2) mt = fmax3(mt, __uint_as_float(sv[i]), __uint_as_float(sv[i + 1]));
          mt *= c;
        } else {
#pragma unroll
          for (int i = 0; i < kBN; ++i) {
            const float f = (i < lim && (i < 64 ? ok_lo : ok_hi)) ? __uint_as_float(sv[i]) * c : -INFINITY;
            sv[i] = __float_as_uint(f);
            mt = fmaxf(mt, f);
          }
        }
        // the reference max moves only when the row max grows by more than
        // the threshold (then p <= 2^threshold below it)
        const float m_new = fmaxf(m, mt);
        const bool need = m_new > m + kRescaleThreshold;
        float alpha = 1.f;
        if (need) {
          alpha = (m == -INFINITY) ? 0.f : ex2_approx(m - m_new);
          l *= alpha;
          m = m_new;
        }
        if (__any_sync(0xffffffffu, need && j > 0)) {
          if (!wait_next()) {
            aborted = true;
            break;
          }
          // move O_t to the new reference maximum
#pragma unroll
          for (int cc = 0; cc < D; cc += 32) {
            uint32_t o[32];
            tmem_ld_32x32b_x32(tO + cc, o);
            tmem_ld_wait_x32(o);
            const uint64_t al2 = f2_pack(alpha, alpha);
#pragma unroll
            for (int i = 0; i < 32; i += 2) {
              const uint64_t v = f2_fma(f2_pack(__uint_as_float(o[i]), __uint_as_float(o[i + 1])), al2, 0ull);
              float lo, hi;
              f2_unpack(v, lo, hi);
              o[i] = __float_as_uint(lo);
              o[i + 1] = __float_as_uint(hi);
            }
            tmem_st_32x32b_x32(tO + cc, o);
          }
        }
        const float mref = (m == -INFINITY) ? 0.f : m;
        uint64_t acc0 = 0ull, acc1 = 0ull;       // packed (+0.0f, +0.0f) row sums
        if (full) {
          const uint64_t nm2 = f2_pack(-mref, -mref);
#pragma unroll
          for (int i = 0; i < kBN / 2; ++i) {
            float x0, x1;
            f2_unpack(f2_fma(f2_pack(__uint_as_float(sv[2 * i]), __uint_as_float(sv[2 * i + 1])), c2, nm2), x0, x1);
            const float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
            if (i & 1)
              acc1 = f2_add(acc1, f2_pack(p0, p1));
            else
              acc0 = f2_add(acc0, f2_pack(p0, p1));
            pall[i] = pack_bf16x2(p0, p1);
          }
        } else {
#pragma unroll
          for (int i = 0; i < kBN / 2; ++i) {
            const float p0 = ex2_approx(__uint_as_float(sv[2 * i]) - mref);
            const float p1 = ex2_approx(__uint_as_float(sv[2 * i + 1]) - mref);
            if (i & 1)
              acc1 = f2_add(acc1, f2_pack(p0, p1));
            else
              acc0 = f2_add(acc0, f2_pack(p0, p1));
            pall[i] = pack_bf16x2(p0, p1);
          }
        }
        {
          float s0, s1;
          f2_unpack(f2_add(acc0, acc1), s0, s1);
          l += s0 + s1;
        }
        if (!wait_next()) {
          aborted = true;
          break;
        }
        // Hand-off: S_t(j+1) into registers, then P_t(j) over its first 64
        // columns (bf16 pairs fill exactly 64 columns).
        if (j + 1 < n) {
          tmem_ld_32x32b_x32(tS + 0, sv + 0);
          tmem_ld_32x32b_x32(tS + 32, sv + 32);
          tmem_ld_32x32b_x32(tS + 64, sv + 64);
          tmem_ld_32x32b_x32(tS + 96, sv + 96);
          tmem_ld_wait_x128(sv);
        }
#pragma unroll
        for (int q = 0; q < 4; ++q) tmem_st_32x32b_x16(tS + uint32_t(q) * 16u, pall + q * 16);
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(p_full(t));
      }

      if (!aborted) {
        u_next = next_unit(k + 1, sq_next, next_ok, true);
        next_ok = __all_sync(0xffffffffu, next_ok);
      }

      // ---------------------------------------------------------- epilogue
      bool have_o = (U.n_tiles > 0) && !aborted;
      if (have_o) {
        const bool ok = mbar_wait(o_done(t), qn & 1, abort_flag, to);
        have_o = __all_sync(0xffffffffu, ok);
        if (!have_o) aborted = true;
        tc_fence_after();
      }
      uint32_t o[D];
      if (have_o) {
#pragma unroll
        for (int cc = 0; cc < D; cc += 32) tmem_ld_32x32b_x32(tO + cc, o + cc);
        if constexpr (D == 128)
          tmem_ld_wait_x128(o);
        else
          tmem_ld_wait_x32(o), tmem_ld_wait_x32(o + 32);
        // O_t has been read: the next unit's first PV may overwrite it
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(o_free(t));
      } else {
#pragma unroll
        for (int i = 0; i < D; ++i) o[i] = 0u;
      }
      const float inv_l = (l > 0.f && have_o) ? 1.f / l : 0.f;
      // A packed Q tile that runs past its sequence (its last rows belong to
      // the next sequence) is written row by row; every other tile goes out
      // through shared memory and one TMA store.
      const bool tile_full = !kPacked || (U.q0 + (t + 1) * p.Mq <= U.Lq);
      if (!aborted && U.has_rows && !tile_full) {
        if (row_ok) {
          __nv_bfloat16* orow =
              p.out + ((size_t(U.qbase) + size_t(token)) * p.Hq + size_t(U.kvh) * p.G + g) * D;
#pragma unroll
          for (int c8 = 0; c8 < D / 8; ++c8) {
            uint4 w;
            w.x = pack_bf16x2(__uint_as_float(o[8 * c8 + 0]) * inv_l, __uint_as_float(o[8 * c8 + 1]) * inv_l);
            w.y = pack_bf16x2(__uint_as_float(o[8 * c8 + 2]) * inv_l, __uint_as_float(o[8 * c8 + 3]) * inv_l);
            w.z = pack_bf16x2(__uint_as_float(o[8 * c8 + 4]) * inv_l, __uint_as_float(o[8 * c8 + 5]) * inv_l);
            w.w = pack_bf16x2(__uint_as_float(o[8 * c8 + 6]) * inv_l, __uint_as_float(o[8 * c8 + 7]) * inv_l);
            *reinterpret_cast<uint4*>(orow + 8 * c8) = w;
          }
        }
      } else if (!aborted && U.has_rows) {
        // Normalised bf16 rows go to a staging block in shared memory, 64
        // columns at a time, and one thread writes each block to global memory
        // with a TMA store (rows of tokens past Sq fall outside the tensor and
        // are not written).  Row r of the block is 128 bytes; its 16-byte chunk
        // c sits at position c ^ (r % 8), the 128-byte swizzle of the map.  The
        // hand-offs use mbarriers with bounded waits (not bar.sync), so a warp
        // that gave up on an earlier wait cannot leave the others blocked.
        const uint32_t stage = base + L::kOffOut + uint32_t(t) * L::kHalfBytes;
        const bool leader = (wq == 0 && lane == 0);
#pragma unroll
        for (int h = 0; h < L::kHalves; ++h) {
          const uint32_t ph = n_stage & 1;
          ++n_stage;
          if (leader) {
            bulk_wait_read_all();        // the previous store has finished reading the block
            mbar_arrive(stg_free(t));
          }
          const bool ok = __all_sync(0xffffffffu, mbar_wait(stg_free(t), ph, abort_flag, to));
          if (ok) {
#pragma unroll
            for (int c8 = 0; c8 < 8; ++c8) {
              uint32_t w[4];
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const int col = h * 64 + c8 * 8 + 2 * e;
                w[e] = pack_bf16x2(__uint_as_float(o[col]) * inv_l, __uint_as_float(o[col + 1]) * inv_l);
              }
              const uint32_t addr = stage + uint32_t(r) * 128u + (uint32_t(c8 ^ (r & 7)) << 4);
              asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(w[0]), "r"(w[1]),
                           "r"(w[2]), "r"(w[3])
                           : "memory");
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(stg_full(t));
          }
          if (leader && ok && mbar_wait(stg_full(t), ph, abort_flag, to)) {
            tma_store_4d(&tmO, stage, h * 64, U.kvh * p.G, U.qbase + U.q0 + t * p.Mq, U.tb);
            bulk_commit_group();
          }
        }
      }
      if (!aborted && row_ok && p.lse) {
        float lg;
        asm("lg2.approx.f32 %0, %1;" : "=f"(lg) : "f"(l));
        const float lse = (l > 0.f && have_o) ? (m + lg) * 0.6931471805599453f : -INFINITY;
        p.lse[(size_t(U.tb) * p.Hq + size_t(U.kvh) * p.G + g) * size_t(p.lse_stride) + size_t(U.qbase) + token] =
            lse;
      }
      if (U.n_tiles > 0) {
        g_tile += U.n_tiles;
        ++qn;
        if (U.n_tiles >= 2) ++n2;
      }
    }
  }

  if (warp < 8 && (warp & 3) == 0 && lane == 0) bulk_wait_all();   // the epilogue's TMA stores
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

}  // namespace prefill
}  // namespace gqa
