// gqa_api.cu -- the C ABI of libgqa (declared in include/gqa.h): argument
// validation, TMA tensor-map encoding, split planning and kernel launches.
// One translation unit holds every kernel so that they share the device
// error word.
#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <algorithm>
#include <atomic>
#include <mutex>

#include <cuda.h>
#include <cuda_runtime.h>

#include "gqa.h"
#include "common.cuh"
#include "prefill_sm103.cuh"
#include "decode_sm103.cuh"
#include "decode_fp8_sm103.cuh"
#include "fp32_check.cuh"
#include "backward_sm103.cuh"

namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr int kMaxDevices = 64;
constexpr int kMaxSplits = 128;

// ----------------------------------------------------------------- helpers
bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int num_sms(int dev) {
  static int cache[kMaxDevices] = {0};
  if (dev < 0 || dev >= kMaxDevices) return 148;
  if (cache[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
    cache[dev] = n;
  }
  return cache[dev];
}

int current_device() {
  int d = 0;
  if (cudaGetDevice(&d) != cudaSuccess) return 0;
  return d;
}

// Limit of every bounded pipeline wait inside the kernels: 2 s, or the value
// of the environment variable GQA_WAIT_TIMEOUT_NS (nanoseconds), read at each
// launch so that a process can shorten it for one call and restore it.
unsigned long long wait_timeout_ns() {
  const char* e = std::getenv("GQA_WAIT_TIMEOUT_NS");
  const unsigned long long t = e ? std::strtoull(e, nullptr, 10) : 0ull;
  return t > 0 ? t : 2000000000ull;
}

// Test hook: a nonzero GQA_TEST_FORCE_TIMEOUT makes the next launches of the
// prefill and backward kernels wait on a barrier nothing arrives on, so that
// their bounded waits run out and the abort paths run (read at each launch).
int force_timeout() {
  const char* e = std::getenv("GQA_TEST_FORCE_TIMEOUT");
  return (e && e[0] && e[0] != '0') ? 1 : 0;
}

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// Work-unit scheduler slots of the prefill and dQ kernels: each launch takes the next
// slot (a claim counter and a finished-CTA counter); the launch's last CTA
// puts the slot back to zero.  Launches that use one slot must not overlap on
// the GPU, which holds unless kSchedSlots launches are in flight at once.
constexpr int kSchedSlots = 64;
__device__ unsigned int g_prefill_sched[2 * kSchedSlots];
std::atomic<unsigned> g_sched_next{0};

unsigned int* sched_slot(int dev) {
  static unsigned int* base[kMaxDevices] = {nullptr};
  static std::mutex mu;
  if (dev < 0 || dev >= kMaxDevices) return nullptr;
  {
    std::lock_guard<std::mutex> lock(mu);
    if (!base[dev]) {
      void* ptr = nullptr;
      if (cudaGetSymbolAddress(&ptr, g_prefill_sched) != cudaSuccess) return nullptr;
      base[dev] = static_cast<unsigned int*>(ptr);
    }
  }
  return base[dev] + 2 * (g_sched_next.fetch_add(1) % kSchedSlots);
}

// 4-D bf16 tensor map over a row-major [d3][d2][d1][d0] array, 128-byte
// swizzle, out-of-bounds elements read as zero.
bool encode_4d_bf16(CUtensorMap* m, const void* base, uint64_t d0, uint64_t d1, uint64_t d2, uint64_t d3,
                    uint32_t b0, uint32_t b1, uint32_t b2, uint32_t b3) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[4] = {d0, d1, d2, d3};
  const cuuint64_t strides[3] = {d0 * 2, d0 * d1 * 2, d0 * d1 * d2 * 2};
  const cuuint32_t box[4] = {b0, b1, b2, b3};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Sets the dynamic shared-memory size once per device and checks that the
// compiled register count is the one the setmaxnreg split was sized for: the
// softmax warpgroups' setmaxnreg.inc can only complete if the block was
// launched with kLaunchRegs registers per thread.
template <int D>
bool prefill_smem_attr_set(int dev) {
  namespace pf = gqa::prefill;
  static bool done[kMaxDevices] = {false};
  if (dev >= 0 && dev < kMaxDevices && done[dev]) return true;
  const int smem = int(pf::Layout<D>::kSmemAlloc);
  static_assert(2 * 128 * pf::kSoftmaxRegs + 128 * pf::kOtherRegs <= pf::kThreads * pf::kLaunchRegs,
                "register split exceeds the launch budget");
  // both layouts: dense and packed
  // every layout: dense, packed, block-sparse
  for (const void* fn : {reinterpret_cast<const void*>(pf::prefill_kernel<D, false, false>),
                         reinterpret_cast<const void*>(pf::prefill_kernel<D, true, false>),
                         reinterpret_cast<const void*>(pf::prefill_kernel<D, false, true>)}) {
    cudaFuncAttributes fa;
    if (cudaFuncGetAttributes(&fa, fn) != cudaSuccess) return false;
    if (fa.numRegs != pf::kLaunchRegs) return false;
    if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess) return false;
  }
  if (dev >= 0 && dev < kMaxDevices) done[dev] = true;
  return true;
}

// Dense layout (cu_q == nullptr): q/out [B, Sq, Hq, D], k/v [B, Sk, Hkv, D].
// Packed layout: q/out [total_q, Hq, D], k/v [total_k, Hkv, D], sequence b at
// rows cu_q[b].. / cu_k[b].., Sq / Sk = the largest sequence lengths.
template <int D>
int launch_prefill_bf16(const void* q, const void* k, const void* v, void* out, float* lse, int B, int Hq, int Hkv,
                        int Sq, int Sk, float scale, int causal, const int* seqlens_k, const int* cu_q,
                        const int* cu_k, int total_q, int total_k, const uint8_t* bmask, int bs,
                        cudaStream_t stream) {
  namespace pf = gqa::prefill;
  const int G = Hq / Hkv;
  const int Mq = pf::kBM / G;
  const long long n_qblk = (Sq + pf::kNQT * Mq - 1) / (pf::kNQT * Mq);
  const long long n_units = n_qblk * B * Hkv;
  if (n_units <= 0 || n_units > 0x7fffffffLL) return GQA_ERR_UNSUPPORTED;
  // persistent grid: one CTA per SM (the kernel's shared memory and register
  // use allow no more), each looping over work units
  const long long grid = std::min<long long>(n_units, num_sms(current_device()));
  CUtensorMap tmQ, tmK, tmV, tmO;
  // packed: the maps see one batch entry of total_q / total_k rows
  const uint64_t mq_rows = cu_q ? uint64_t(total_q) : uint64_t(Sq);
  const uint64_t mk_rows = cu_q ? uint64_t(total_k) : uint64_t(Sk);
  const uint64_t m_batch = cu_q ? 1u : uint64_t(B);
  if (!encode_4d_bf16(&tmQ, q, D, Hq, mq_rows, m_batch, 64, G, Mq, 1) ||
      !encode_4d_bf16(&tmK, k, D, Hkv, mk_rows, m_batch, 64, 1, 128, 1) ||
      !encode_4d_bf16(&tmV, v, D, Hkv, mk_rows, m_batch, 64, 1, 128, 1) ||
      !encode_4d_bf16(&tmO, out, D, Hq, mq_rows, m_batch, 64, G, Mq, 1))
    return GQA_ERR_CUDA;
  if (!prefill_smem_attr_set<D>(current_device())) return GQA_ERR_CUDA;
  pf::Params p{};
  p.out = static_cast<__nv_bfloat16*>(out);
  p.lse = lse;
  p.seqlens = cu_q ? nullptr : seqlens_k;
  p.cu_q = cu_q;
  p.cu_k = cu_q ? cu_k : nullptr;
  p.total_q = total_q;
  p.total_k = total_k;
  p.lse_stride = cu_q ? total_q : Sq;
  p.bmask = bmask;
  p.bs = bs;
  p.n_qb = bmask ? (Sq + bs - 1) / bs : 0;
  p.n_kb = bmask ? (Sk + bs - 1) / bs : 0;
  p.B = B;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.G = G;
  p.Sq = Sq;
  p.Sk = Sk;
  p.Mq = Mq;
  p.n_qblk = int(n_qblk);
  p.n_units = int(n_units);
  p.sched = sched_slot(current_device());
  if (!p.sched) return GQA_ERR_CUDA;
  p.causal = causal ? 1 : 0;
  p.scale_log2 = scale * kLog2e;
  p.timeout_ns = wait_timeout_ns();
  p.test_stall = force_timeout();
  if (bmask)
    pf::prefill_kernel<D, false, true><<<unsigned(grid), pf::kThreads, pf::Layout<D>::kSmemAlloc, stream>>>(
        tmQ, tmK, tmV, tmO, p);
  else if (cu_q)
    pf::prefill_kernel<D, true, false><<<unsigned(grid), pf::kThreads, pf::Layout<D>::kSmemAlloc, stream>>>(tmQ, tmK, tmV,
                                                                                                 tmO, p);
  else
    pf::prefill_kernel<D, false, false><<<unsigned(grid), pf::kThreads, pf::Layout<D>::kSmemAlloc, stream>>>(tmQ, tmK, tmV,
                                                                                                  tmO, p);
  return cudaGetLastError() == cudaSuccess ? GQA_OK : GQA_ERR_CUDA;
}

// Dynamic shared memory of the decode split kernel: the warps' cp.async
// rings, reused for the final merge of the warps.
template <int D>
constexpr int decode_smem_bytes() {
  namespace dc = gqa::decode;
  constexpr int ring = int(dc::Ring<D>::kBytes);
  constexpr int merge = int(sizeof(float)) * (dc::kWarps * 8 * D + 2 * dc::kWarps * 8);
  return ring > merge ? ring : merge;
}

bool decode_smem_attr_set(int dev) {
  static bool done[kMaxDevices] = {false};
  if (dev >= 0 && dev < kMaxDevices && done[dev]) return true;
  if (cudaFuncSetAttribute(gqa::decode::decode_split_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           decode_smem_bytes<64>()) != cudaSuccess ||
      cudaFuncSetAttribute(gqa::decode::decode_split_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           decode_smem_bytes<128>()) != cudaSuccess)
    return false;
  if (dev >= 0 && dev < kMaxDevices) done[dev] = true;
  return true;
}

bool decode_fp8_smem_attr_set(int dev) {
  static bool done[kMaxDevices] = {false};
  if (dev >= 0 && dev < kMaxDevices && done[dev]) return true;
  if (cudaFuncSetAttribute(gqa::decode::decode_split_fp8_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           int(gqa::decode::RingF8::kBytes)) != cudaSuccess)
    return false;
  if (dev >= 0 && dev < kMaxDevices) done[dev] = true;
  return true;
}

template <int D>
bool bwd_smem_attr_set(int dev) {
  namespace bw = gqa::bwd;
  static bool done[kMaxDevices] = {false};
  if (dev >= 0 && dev < kMaxDevices && done[dev]) return true;
  if (cudaFuncSetAttribute(bw::dq_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           int(bw::DqLayout<D>::kSmemAlloc)) != cudaSuccess ||
      cudaFuncSetAttribute(bw::dkdv_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           int(bw::KvLayout<D>::kSmemAlloc)) != cudaSuccess)
    return false;
  if (dev >= 0 && dev < kMaxDevices) done[dev] = true;
  return true;
}

// Dsum, then dQ and dK/dV (independent of each other) on one stream.
// Side stream of the backward, per device: dK/dV runs on it beside dQ, so
// that its CTAs take the SMs that dQ's persistent CTAs leave as they finish
// (and dQ's last CTAs run beside dK/dV's last wave) instead of the two
// kernels each ending on a partly idle GPU.
struct BwdAux {
  bool ready = false;
  cudaStream_t st = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr;
};
std::mutex g_bwd_aux_mu;
BwdAux g_bwd_aux[kMaxDevices];

// q, out, dout [B, Sq, Hq, D]; k, v [B, Sk, Hkv, D] (bf16).
template <int D>
int launch_bwd(gqa::bwd::Params p, const void* q, const void* k, const void* v, cudaStream_t stream) {
  namespace bw = gqa::bwd;
  const int Mq = 128 / p.G;
  p.Mq = Mq;
  p.n_qt = (p.Sq + Mq - 1) / Mq;
  p.n_kt = (p.Sk + bw::kBN - 1) / bw::kBN;
  p.scale_log2 = p.scale * kLog2e;
  p.timeout_ns = wait_timeout_ns();
  p.test_stall = force_timeout();
  // dq_kernel: Q / dO tiles of Mq tokens x G heads (row = token * G + head),
  // K / V tiles of 128 keys; dkdv_kernel: Q / dO tiles of 128 tokens of one
  // head, K / V tiles of 128 keys.
  CUtensorMap tmQg, tmDOg, tmQ1, tmDO1, tmK, tmV;
  if (!encode_4d_bf16(&tmQg, q, D, p.Hq, p.Sq, p.B, 64, p.G, Mq, 1) ||
      !encode_4d_bf16(&tmDOg, p.dout, D, p.Hq, p.Sq, p.B, 64, p.G, Mq, 1) ||
      !encode_4d_bf16(&tmQ1, q, D, p.Hq, p.Sq, p.B, 64, 1, bw::kBQ, 1) ||
      !encode_4d_bf16(&tmDO1, p.dout, D, p.Hq, p.Sq, p.B, 64, 1, bw::kBQ, 1) ||
      !encode_4d_bf16(&tmK, k, D, p.Hkv, p.Sk, p.B, 64, 1, bw::kBN, 1) ||
      !encode_4d_bf16(&tmV, v, D, p.Hkv, p.Sk, p.B, 64, 1, bw::kBN, 1))
    return GQA_ERR_CUDA;
  if (!bwd_smem_attr_set<D>(current_device())) return GQA_ERR_CUDA;
  const long long dsum_threads = (long long)p.B * p.Hq * p.Sq * (D / 8);
  bw::dsum_kernel<D><<<unsigned((dsum_threads + 255) / 256), 256, 0, stream>>>(p);
  // dq_kernel is persistent: at most one CTA per SM, each looping over tiles
  const long long dq_tiles = (long long)p.n_qt * p.Hkv * p.B;
  if (dq_tiles > 0x7fffffffLL) return GQA_ERR_UNSUPPORTED;
  const unsigned gq = unsigned(std::min<long long>(dq_tiles, num_sms(current_device())));
  const dim3 gk(unsigned(p.n_kt), unsigned(p.Hkv), unsigned(p.B));
  const int dev = current_device();
  if (dev < 0 || dev >= kMaxDevices) return GQA_ERR_CUDA;
  p.sched = sched_slot(dev);
  if (!p.sched) return GQA_ERR_CUDA;
  // Fork after Dsum: dK/dV on the caller's stream, launched first, and dQ on
  // the side stream: its persistent CTAs take SMs as dK/dV's CTAs leave them
  // and claim tiles as they go, so the last partial wave of dK/dV and dQ's
  // work share the GPU.  The caller's stream then waits for both.  The lock
  // keeps the record / wait pairs of concurrent callers apart (the events
  // are shared).
  std::lock_guard<std::mutex> lock(g_bwd_aux_mu);
  BwdAux& ax = g_bwd_aux[dev];
  if (!ax.ready) {
    if (cudaStreamCreateWithFlags(&ax.st, cudaStreamNonBlocking) != cudaSuccess ||
        cudaEventCreateWithFlags(&ax.fork, cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&ax.join, cudaEventDisableTiming) != cudaSuccess)
      return GQA_ERR_CUDA;
    ax.ready = true;
  }
  if (cudaEventRecord(ax.fork, stream) != cudaSuccess || cudaStreamWaitEvent(ax.st, ax.fork, 0) != cudaSuccess)
    return GQA_ERR_CUDA;
  bw::dkdv_kernel<D><<<gk, bw::kThreads, bw::KvLayout<D>::kSmemAlloc, stream>>>(tmK, tmV, tmQ1, tmDO1, p);
  bw::dq_kernel<D><<<gq, bw::kThreads, bw::DqLayout<D>::kSmemAlloc, ax.st>>>(tmQg, tmDOg, tmK, tmV, p);
  if (cudaGetLastError() != cudaSuccess) return GQA_ERR_CUDA;
  if (cudaEventRecord(ax.join, ax.st) != cudaSuccess || cudaStreamWaitEvent(stream, ax.join, 0) != cudaSuccess)
    return GQA_ERR_CUDA;
  return GQA_OK;
}

int launch_f32(const gqa::f32::Params& p, cudaStream_t stream) {
  const long long rows = p.cu_q ? (long long)p.Hq * p.total_q : (long long)p.B * p.Hq * p.Sq;
  const long long gx = (rows + gqa::f32::kWarps - 1) / gqa::f32::kWarps;
  if (gx > 0x7fffffffLL || p.nsplit > 65535) return GQA_ERR_UNSUPPORTED;
  gqa::f32::attention_kernel<<<dim3(unsigned(gx), unsigned(p.nsplit)), gqa::f32::kWarps * 32, 0, stream>>>(p);
  return cudaGetLastError() == cudaSuccess ? GQA_OK : GQA_ERR_CUDA;
}

struct SplitPlan {
  int n;          // number of splits actually launched
  int len;        // keys per split (multiple of 16)
};

// n requested (<= 0: automatic) -> split length rounded up to 16 keys; the
// launched count is ceil(Smax / len) so that no split is empty for a full cache.
// Automatic: about target_len keys per split, and enough CTAs (B * ceil(Hkv /
// heads_per_cta) per split) for several waves.  The bf16 / fp32 split kernel
// takes 1024 keys of one K/V head per CTA; the FP8 kernel, whose CTAs stream
// four K/V heads at half the bytes per key, 512 keys (measured on B300 for
// llama_decode_fp8: 512 keys per split 0.126 ms, 1024 keys 0.139 ms).
SplitPlan plan_splits(int B, int Hkv, int Smax, int num_splits, int target_len = 1024, int heads_per_cta = 1) {
  int n = num_splits;
  if (n <= 0) {
    const int sms = num_sms(current_device());
    n = (Smax + target_len - 1) / target_len;
    const long long want = 4LL * sms;
    const long long groups = (long long)B * ((Hkv + heads_per_cta - 1) / heads_per_cta);
    while ((long long)n * groups < want && n < kMaxSplits && (Smax + n) / (n + 1) >= 256) ++n;
  }
  n = std::max(1, std::min(n, kMaxSplits));
  const int blocks = (Smax + 15) / 16;
  n = std::min(n, blocks);
  int len = (Smax + n - 1) / n;
  len = (len + 15) / 16 * 16;
  SplitPlan sp;
  sp.len = len;
  sp.n = (Smax + len - 1) / len;
  return sp;
}

SplitPlan plan_splits_fp8(int B, int Hkv, int Smax, int num_splits) {
  return plan_splits(B, Hkv, Smax, num_splits, 512, gqa::decode::kF8Warps);
}

size_t workspace_for(int B, int Hq, int D, int n) {
  if (n <= 1) return 0;
  const size_t o = size_t(B) * Hq * n * D * sizeof(float);
  const size_t l = size_t(B) * Hq * n * sizeof(float);
  return ((o + 255) / 256) * 256 + l;
}

// The split-KV combine, launched as a programmatic dependent of the split
// kernel just queued on the same stream: its launch overlaps the split
// kernel's tail, and griddepcontrol.wait inside it orders the reads of the
// partials after that grid has completed.
template <typename OutT, int VEC>
cudaError_t launch_combine(cudaStream_t st, const float* part_o, const float* part_lse, const int* seqlens, OutT* out,
                           int B, int Hq, int D, int nsplit, int split_len, int Smax) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned((B * Hq + 3) / 4));
  cfg.blockDim = dim3(128);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, gqa::decode::combine_kernel<OutT, VEC>, part_o, part_lse, seqlens, out, B, Hq, D,
                            nsplit, split_len, Smax);
}

}  // namespace


// ====================================================================== ABI
extern "C" {

const char* gqa_status_string(int status) {
  switch (status) {
    case GQA_OK: return "GQA_OK";
    case GQA_ERR_INVALID_ARG: return "GQA_ERR_INVALID_ARG";
    case GQA_ERR_UNSUPPORTED: return "GQA_ERR_UNSUPPORTED";
    case GQA_ERR_CUDA: return "GQA_ERR_CUDA";
    case GQA_ERR_DEVICE_TIMEOUT: return "GQA_ERR_DEVICE_TIMEOUT";
    case GQA_ERR_DEVICE_BOUNDS: return "GQA_ERR_DEVICE_BOUNDS";
    default: return "GQA_ERR_UNKNOWN";
  }
}

}  // extern "C"

namespace {

// Argument checks of gqa_fwd: GQA_OK when the call would launch its kernel.
int fwd_arg_status(const void* q, const void* k, const void* v, const void* out, const float* lse, int B, int Hq,
                   int Hkv, int Sq, int Sk, int D, float scale, int causal, const int* seqlens_k, int dtype) {
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || Sq <= 0 || Sk <= 0 || D <= 0) return GQA_ERR_INVALID_ARG;
  if (Hq % Hkv != 0) return GQA_ERR_INVALID_ARG;
  if (!q || !k || !v || !out) return GQA_ERR_INVALID_ARG;
  if (!std::isfinite(scale)) return GQA_ERR_INVALID_ARG;
  if (causal != 0 && causal != 1) return GQA_ERR_INVALID_ARG;
  if ((lse && !aligned(lse, 4)) || (seqlens_k && !aligned(seqlens_k, 4))) return GQA_ERR_INVALID_ARG;
  if (dtype == GQA_DTYPE_BF16) {
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(out, 16)) return GQA_ERR_INVALID_ARG;
    if (D != 64 && D != 128) return GQA_ERR_UNSUPPORTED;
    if (Hq / Hkv > gqa::prefill::kBM) return GQA_ERR_UNSUPPORTED;
    if ((long long)Hq * D * Sq * B > (1LL << 40)) return GQA_ERR_UNSUPPORTED;
    return GQA_OK;
  }
  if (dtype == GQA_DTYPE_FP32) {
    if (!aligned(q, 4) || !aligned(k, 4) || !aligned(v, 4) || !aligned(out, 4)) return GQA_ERR_INVALID_ARG;
    if (D > gqa::f32::kMaxD) return GQA_ERR_UNSUPPORTED;
    return GQA_OK;
  }
  return GQA_ERR_INVALID_ARG;
}

}  // namespace

extern "C" {

int gqa_fwd(const void* q, const void* k, const void* v, void* out, float* lse, int B, int Hq, int Hkv, int Sq,
            int Sk, int D, float scale, int causal, const int* seqlens_k, int dtype, void* stream) {
  const int arg = fwd_arg_status(q, k, v, out, lse, B, Hq, Hkv, Sq, Sk, D, scale, causal, seqlens_k, dtype);
  if (arg != GQA_OK) return arg;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (dtype == GQA_DTYPE_BF16) {
    return D == 64 ? launch_prefill_bf16<64>(q, k, v, out, lse, B, Hq, Hkv, Sq, Sk, scale, causal, seqlens_k,
                                             nullptr, nullptr, 0, 0, nullptr, 0, st)
                   : launch_prefill_bf16<128>(q, k, v, out, lse, B, Hq, Hkv, Sq, Sk, scale, causal, seqlens_k,
                                              nullptr, nullptr, 0, 0, nullptr, 0, st);
  }
  {
    gqa::f32::Params p{};
    p.q = static_cast<const float*>(q);
    p.k = static_cast<const float*>(k);
    p.v = static_cast<const float*>(v);
    p.out = static_cast<float*>(out);
    p.lse = lse;
    p.seqlens = seqlens_k;
    p.q_sb = (long long)Sq * Hq * D;
    p.q_ss = (long long)Hq * D;
    p.q_sh = D;
    p.k_sb = (long long)Sk * Hkv * D;
    p.k_ss = (long long)Hkv * D;
    p.k_sh = D;
    p.B = B;
    p.Hq = Hq;
    p.Hkv = Hkv;
    p.G = Hq / Hkv;
    p.Sq = Sq;
    p.Sk = Sk;
    p.D = D;
    p.causal = causal;
    p.scale = scale;
    p.nsplit = 1;
    p.split_len = Sk;
    p.len_cap = Sk;
    return launch_f32(p, st);
  }
}

}  // extern "C"

// ===================================================== host-buffer prefill
// Copy streams and events of gqa_fwd_host, created once per device.
namespace {

constexpr int kHostPipeMaxChunks = 64;

struct HostPipe {
  bool ready = false;
  cudaStream_t in = nullptr, out = nullptr;
  cudaEvent_t start = nullptr, done = nullptr;
  cudaEvent_t in_done[kHostPipeMaxChunks] = {};
  cudaEvent_t comp_done[kHostPipeMaxChunks] = {};
};

std::mutex g_host_pipe_mu;
HostPipe g_host_pipe[kMaxDevices];

HostPipe* host_pipe(int dev) {
  if (dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_host_pipe_mu);
  HostPipe& hp = g_host_pipe[dev];
  if (!hp.ready) {
    const unsigned ev = cudaEventDisableTiming;
    bool ok = cudaStreamCreateWithFlags(&hp.in, cudaStreamNonBlocking) == cudaSuccess &&
              cudaStreamCreateWithFlags(&hp.out, cudaStreamNonBlocking) == cudaSuccess &&
              cudaEventCreateWithFlags(&hp.start, ev) == cudaSuccess &&
              cudaEventCreateWithFlags(&hp.done, ev) == cudaSuccess;
    for (int i = 0; ok && i < kHostPipeMaxChunks; ++i)
      ok = cudaEventCreateWithFlags(&hp.in_done[i], ev) == cudaSuccess &&
           cudaEventCreateWithFlags(&hp.comp_done[i], ev) == cudaSuccess;
    if (!ok) return nullptr;
    hp.ready = true;
  }
  return &hp;
}

}  // namespace

extern "C" {

int gqa_fwd_host(const void* q_h, const void* k_h, const void* v_h, void* out_h, float* lse_h, int B, int Hq,
                 int Hkv, int Sq, int Sk, int D, float scale, int causal, const int* seqlens_k_h, int dtype,
                 void* q_d, void* k_d, void* v_d, void* out_d, float* lse_d, int* seqlens_d, int chunk_b,
                 void* stream) {
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || Sq <= 0 || Sk <= 0 || D <= 0) return GQA_ERR_INVALID_ARG;
  if (!q_h || !k_h || !v_h || !out_h || !q_d || !k_d || !v_d || !out_d) return GQA_ERR_INVALID_ARG;
  if ((lse_h == nullptr) != (lse_d == nullptr)) return GQA_ERR_INVALID_ARG;
  if ((seqlens_k_h == nullptr) != (seqlens_d == nullptr)) return GQA_ERR_INVALID_ARG;
  // the whole call's arguments, as gqa_fwd checks them, before anything is
  // enqueued (every chunk then passes the same checks)
  const int arg = fwd_arg_status(q_d, k_d, v_d, out_d, lse_d, B, Hq, Hkv, Sq, Sk, D, scale, causal, seqlens_d, dtype);
  if (arg != GQA_OK) return arg;
  const size_t esz = dtype == GQA_DTYPE_BF16 ? 2 : 4;
  int cb = chunk_b > 0 ? chunk_b : std::max(1, B / 8);
  cb = std::max(cb, (B + kHostPipeMaxChunks - 1) / kHostPipeMaxChunks);   // at most kHostPipeMaxChunks chunks
  cb = std::min(cb, B);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  HostPipe* hp = host_pipe(current_device());
  if (!hp) return GQA_ERR_CUDA;
  // per batch entry
  const size_t qb = size_t(Sq) * Hq * D * esz, kb = size_t(Sk) * Hkv * D * esz, lb = size_t(Hq) * Sq * 4;
  auto c8 = [](const void* p, size_t off) { return static_cast<const char*>(p) + off; };
  auto m8 = [](void* p, size_t off) { return static_cast<char*>(p) + off; };
  // the copy streams start after the work already enqueued on `stream`
  if (cudaEventRecord(hp->start, st) != cudaSuccess || cudaStreamWaitEvent(hp->in, hp->start, 0) != cudaSuccess ||
      cudaStreamWaitEvent(hp->out, hp->start, 0) != cudaSuccess)
    return GQA_ERR_CUDA;
  int rc = GQA_OK;
  int ci = 0;
  for (int b0 = 0; b0 < B; b0 += cb, ++ci) {
    const int nb = std::min(cb, B - b0);
    // inputs of the chunk: host -> device
    if (cudaMemcpyAsync(m8(q_d, b0 * qb), c8(q_h, b0 * qb), nb * qb, cudaMemcpyHostToDevice, hp->in) != cudaSuccess ||
        cudaMemcpyAsync(m8(k_d, b0 * kb), c8(k_h, b0 * kb), nb * kb, cudaMemcpyHostToDevice, hp->in) != cudaSuccess ||
        cudaMemcpyAsync(m8(v_d, b0 * kb), c8(v_h, b0 * kb), nb * kb, cudaMemcpyHostToDevice, hp->in) != cudaSuccess ||
        (seqlens_d && cudaMemcpyAsync(seqlens_d + b0, seqlens_k_h + b0, nb * sizeof(int), cudaMemcpyHostToDevice,
                                      hp->in) != cudaSuccess) ||
        cudaEventRecord(hp->in_done[ci], hp->in) != cudaSuccess ||
        cudaStreamWaitEvent(st, hp->in_done[ci], 0) != cudaSuccess) {
      rc = GQA_ERR_CUDA;
      break;
    }
    // the chunk's attention on `stream`
    rc = gqa_fwd(c8(q_d, b0 * qb), c8(k_d, b0 * kb), c8(v_d, b0 * kb), m8(out_d, b0 * qb),
                 lse_d ? reinterpret_cast<float*>(m8(lse_d, b0 * lb)) : nullptr, nb, Hq, Hkv, Sq, Sk, D, scale, causal,
                 seqlens_d ? seqlens_d + b0 : nullptr, dtype, stream);
    if (rc != GQA_OK) break;
    // outputs of the chunk: device -> host
    if (cudaEventRecord(hp->comp_done[ci], st) != cudaSuccess ||
        cudaStreamWaitEvent(hp->out, hp->comp_done[ci], 0) != cudaSuccess ||
        cudaMemcpyAsync(m8(out_h, b0 * qb), c8(out_d, b0 * qb), nb * qb, cudaMemcpyDeviceToHost, hp->out) !=
            cudaSuccess ||
        (lse_d && cudaMemcpyAsync(m8(lse_h, b0 * lb), c8(lse_d, b0 * lb), nb * lb, cudaMemcpyDeviceToHost, hp->out) !=
                      cudaSuccess)) {
      rc = GQA_ERR_CUDA;
      break;
    }
  }
  // `stream` completes only after the last copy (also after a failure part-way)
  if (cudaEventRecord(hp->done, hp->out) != cudaSuccess || cudaStreamWaitEvent(st, hp->done, 0) != cudaSuccess)
    return GQA_ERR_CUDA;
  return rc;
}

int gqa_fwd_varlen(const void* q, const void* k, const void* v, void* out, float* lse, const int* cu_seqlens_q,
                   const int* cu_seqlens_k, int B, int Hq, int Hkv, int max_seqlen_q, int max_seqlen_k, int total_q,
                   int total_k, int D, float scale, int causal, int dtype, void* stream) {
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || D <= 0 || max_seqlen_q <= 0 || max_seqlen_k <= 0 || total_q <= 0 ||
      total_k <= 0)
    return GQA_ERR_INVALID_ARG;
  if (Hq % Hkv != 0) return GQA_ERR_INVALID_ARG;
  if (!q || !k || !v || !out || !cu_seqlens_q || !cu_seqlens_k) return GQA_ERR_INVALID_ARG;
  if (!aligned(cu_seqlens_q, 4) || !aligned(cu_seqlens_k, 4) || (lse && !aligned(lse, 4))) return GQA_ERR_INVALID_ARG;
  if (!std::isfinite(scale)) return GQA_ERR_INVALID_ARG;
  if (causal != 0 && causal != 1) return GQA_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (dtype == GQA_DTYPE_BF16) {
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(out, 16)) return GQA_ERR_INVALID_ARG;
    if (D != 64 && D != 128) return GQA_ERR_UNSUPPORTED;
    if (Hq / Hkv > gqa::prefill::kBM) return GQA_ERR_UNSUPPORTED;
    if ((long long)Hq * D * total_q > (1LL << 40) || (long long)Hkv * D * total_k > (1LL << 40))
      return GQA_ERR_UNSUPPORTED;
    return D == 64 ? launch_prefill_bf16<64>(q, k, v, out, lse, B, Hq, Hkv, max_seqlen_q, max_seqlen_k, scale,
                                             causal, nullptr, cu_seqlens_q, cu_seqlens_k, total_q, total_k,
                                             nullptr, 0, st)
                   : launch_prefill_bf16<128>(q, k, v, out, lse, B, Hq, Hkv, max_seqlen_q, max_seqlen_k, scale,
                                              causal, nullptr, cu_seqlens_q, cu_seqlens_k, total_q, total_k,
                                              nullptr, 0, st);
  }
  if (dtype == GQA_DTYPE_FP32) {
    if (!aligned(q, 4) || !aligned(k, 4) || !aligned(v, 4) || !aligned(out, 4)) return GQA_ERR_INVALID_ARG;
    if (D > gqa::f32::kMaxD) return GQA_ERR_UNSUPPORTED;
    gqa::f32::Params p{};
    p.q = static_cast<const float*>(q);
    p.k = static_cast<const float*>(k);
    p.v = static_cast<const float*>(v);
    p.out = static_cast<float*>(out);
    p.lse = lse;
    p.cu_q = cu_seqlens_q;
    p.cu_k = cu_seqlens_k;
    p.total_q = total_q;
    p.total_k = total_k;
    p.q_ss = (long long)Hq * D;
    p.q_sh = D;
    p.k_ss = (long long)Hkv * D;
    p.k_sh = D;
    p.B = B;
    p.Hq = Hq;
    p.Hkv = Hkv;
    p.G = Hq / Hkv;
    p.Sq = max_seqlen_q;
    p.Sk = max_seqlen_k;
    p.D = D;
    p.causal = causal;
    p.scale = scale;
    p.nsplit = 1;
    p.split_len = max_seqlen_k;
    p.len_cap = max_seqlen_k;
    return launch_f32(p, st);
  }
  return GQA_ERR_INVALID_ARG;
}

int gqa_decode_fp8(const void* q, const void* kcache, const void* vcache, const int* cache_seqlens, void* out,
                   int B, int Hq, int Hkv, int D, float scale, float k_scale, float v_scale, int num_splits,
                   int max_seqlen_k, void* workspace, size_t workspace_bytes, void* stream) {
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || D <= 0 || max_seqlen_k <= 0) return GQA_ERR_INVALID_ARG;
  if (Hq % Hkv != 0 || num_splits > kMaxSplits) return GQA_ERR_INVALID_ARG;
  if (!q || !kcache || !vcache || !cache_seqlens || !out) return GQA_ERR_INVALID_ARG;
  if (!std::isfinite(scale) || !std::isfinite(k_scale) || !std::isfinite(v_scale) || !aligned(cache_seqlens, 4))
    return GQA_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(kcache, 16) || !aligned(vcache, 16) || !aligned(out, 16)) return GQA_ERR_INVALID_ARG;
  const int G = Hq / Hkv;
  if (D != gqa::decode::kF8D || G > 8) return GQA_ERR_UNSUPPORTED;
  if (B > 65535 || Hkv > 65535) return GQA_ERR_UNSUPPORTED;
  const SplitPlan sp = plan_splits_fp8(B, Hkv, max_seqlen_k, num_splits);
  const size_t need = workspace_for(B, Hq, D, sp.n);
  if (need > 0 && (!workspace || workspace_bytes < need || !aligned(workspace, 16))) return GQA_ERR_INVALID_ARG;
  float* part_o = static_cast<float*>(workspace);
  float* part_lse = need ? reinterpret_cast<float*>(static_cast<char*>(workspace) +
                                                    ((size_t(B) * Hq * sp.n * D * sizeof(float) + 255) / 256) * 256)
                         : nullptr;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  gqa::decode::ParamsF8 p;
  p.q = static_cast<const __nv_bfloat16*>(q);
  p.kc = static_cast<const uint8_t*>(kcache);
  p.vc = static_cast<const uint8_t*>(vcache);
  p.seqlens = cache_seqlens;
  p.out = static_cast<__nv_bfloat16*>(out);
  p.part_o = part_o;
  p.part_lse = part_lse;
  p.B = B;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.G = G;
  p.Smax = max_seqlen_k;
  p.nsplit = sp.n;
  p.split_len = sp.len;
  p.scale_k_log2 = float(double(scale) * double(k_scale) * 1.4426950408889634);
  p.v_scale = v_scale;
  if (!decode_fp8_smem_attr_set(current_device())) return GQA_ERR_CUDA;
  gqa::decode::decode_split_fp8_kernel<<<dim3(sp.n, (Hkv + gqa::decode::kF8Warps - 1) / gqa::decode::kF8Warps, B),
                                         gqa::decode::kF8Threads, gqa::decode::RingF8::kBytes,
                                         st>>>(p);
  if (cudaGetLastError() != cudaSuccess) return GQA_ERR_CUDA;
  if (sp.n > 1 && launch_combine<__nv_bfloat16, 4>(st, part_o, part_lse, cache_seqlens, static_cast<__nv_bfloat16*>(out),
                                                    B, Hq, D, sp.n, sp.len, max_seqlen_k) != cudaSuccess)
    return GQA_ERR_CUDA;
  return GQA_OK;
}

int gqa_fwd_sparse(const void* q, const void* k, const void* v, void* out, float* lse, const unsigned char* block_mask,
                   int block_size, int B, int Hq, int Hkv, int Sq, int Sk, int D, float scale, int causal,
                   const int* seqlens_k, int dtype, void* stream) {
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || Sq <= 0 || Sk <= 0 || D <= 0) return GQA_ERR_INVALID_ARG;
  if (Hq % Hkv != 0) return GQA_ERR_INVALID_ARG;
  if (!q || !k || !v || !out || !block_mask) return GQA_ERR_INVALID_ARG;
  if (block_size != 64 && block_size != 128) return GQA_ERR_INVALID_ARG;
  if (!std::isfinite(scale)) return GQA_ERR_INVALID_ARG;
  if (causal != 0 && causal != 1) return GQA_ERR_INVALID_ARG;
  if ((lse && !aligned(lse, 4)) || (seqlens_k && !aligned(seqlens_k, 4))) return GQA_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (dtype == GQA_DTYPE_BF16) {
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(out, 16)) return GQA_ERR_INVALID_ARG;
    if (D != 64 && D != 128) return GQA_ERR_UNSUPPORTED;
    if (Hq / Hkv > gqa::prefill::kBM) return GQA_ERR_UNSUPPORTED;
    if (Sk > 64 * gqa::prefill::kBN) return GQA_ERR_UNSUPPORTED;   // one 64-bit word of key tiles per unit
    if ((long long)Hq * D * Sq * B > (1LL << 40)) return GQA_ERR_UNSUPPORTED;
    return D == 64 ? launch_prefill_bf16<64>(q, k, v, out, lse, B, Hq, Hkv, Sq, Sk, scale, causal, seqlens_k,
                                             nullptr, nullptr, 0, 0, block_mask, block_size, st)
                   : launch_prefill_bf16<128>(q, k, v, out, lse, B, Hq, Hkv, Sq, Sk, scale, causal, seqlens_k,
                                              nullptr, nullptr, 0, 0, block_mask, block_size, st);
  }
  if (dtype == GQA_DTYPE_FP32) {
    if (!aligned(q, 4) || !aligned(k, 4) || !aligned(v, 4) || !aligned(out, 4)) return GQA_ERR_INVALID_ARG;
    if (D > gqa::f32::kMaxD) return GQA_ERR_UNSUPPORTED;
    gqa::f32::Params p{};
    p.q = static_cast<const float*>(q);
    p.k = static_cast<const float*>(k);
    p.v = static_cast<const float*>(v);
    p.out = static_cast<float*>(out);
    p.lse = lse;
    p.seqlens = seqlens_k;
    p.bmask = block_mask;
    p.bs = block_size;
    p.n_kb = (Sk + block_size - 1) / block_size;
    p.q_sb = (long long)Sq * Hq * D;
    p.q_ss = (long long)Hq * D;
    p.q_sh = D;
    p.k_sb = (long long)Sk * Hkv * D;
    p.k_ss = (long long)Hkv * D;
    p.k_sh = D;
    p.B = B;
    p.Hq = Hq;
    p.Hkv = Hkv;
    p.G = Hq / Hkv;
    p.Sq = Sq;
    p.Sk = Sk;
    p.D = D;
    p.causal = causal;
    p.scale = scale;
    p.nsplit = 1;
    p.split_len = Sk;
    p.len_cap = Sk;
    return launch_f32(p, st);
  }
  return GQA_ERR_INVALID_ARG;
}

int gqa_decode_num_splits(int B, int Hkv, int max_seqlen_k, int num_splits) {
  if (B <= 0 || Hkv <= 0 || max_seqlen_k <= 0) return -GQA_ERR_INVALID_ARG;
  if (num_splits > kMaxSplits) return -GQA_ERR_INVALID_ARG;
  return plan_splits(B, Hkv, max_seqlen_k, num_splits).n;
}

size_t gqa_decode_workspace_bytes(int B, int Hq, int Hkv, int D, int num_splits, int max_seqlen_k) {
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || D <= 0 || max_seqlen_k <= 0 || num_splits > kMaxSplits) return 0;
  return workspace_for(B, Hq, D, plan_splits(B, Hkv, max_seqlen_k, num_splits).n);
}

int gqa_decode_fp8_num_splits(int B, int Hkv, int max_seqlen_k, int num_splits) {
  if (B <= 0 || Hkv <= 0 || max_seqlen_k <= 0) return -GQA_ERR_INVALID_ARG;
  if (num_splits > kMaxSplits) return -GQA_ERR_INVALID_ARG;
  return plan_splits_fp8(B, Hkv, max_seqlen_k, num_splits).n;
}

size_t gqa_decode_fp8_workspace_bytes(int B, int Hq, int Hkv, int D, int num_splits, int max_seqlen_k) {
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || D <= 0 || max_seqlen_k <= 0 || num_splits > kMaxSplits) return 0;
  return workspace_for(B, Hq, D, plan_splits_fp8(B, Hkv, max_seqlen_k, num_splits).n);
}

int gqa_decode(const void* q, const void* kcache, const void* vcache, const int* cache_seqlens, void* out, int B,
               int Hq, int Hkv, int D, float scale, int num_splits, int max_seqlen_k, int dtype, void* workspace,
               size_t workspace_bytes, void* stream) {
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || D <= 0 || max_seqlen_k <= 0) return GQA_ERR_INVALID_ARG;
  if (Hq % Hkv != 0 || num_splits > kMaxSplits) return GQA_ERR_INVALID_ARG;
  if (!q || !kcache || !vcache || !cache_seqlens || !out) return GQA_ERR_INVALID_ARG;
  if (!std::isfinite(scale) || !aligned(cache_seqlens, 4)) return GQA_ERR_INVALID_ARG;
  const SplitPlan sp = plan_splits(B, Hkv, max_seqlen_k, num_splits);
  const size_t need = workspace_for(B, Hq, D, sp.n);
  if (need > 0 && (!workspace || workspace_bytes < need || !aligned(workspace, 16))) return GQA_ERR_INVALID_ARG;
  float* part_o = static_cast<float*>(workspace);
  float* part_lse = need ? reinterpret_cast<float*>(static_cast<char*>(workspace) +
                                                    ((size_t(B) * Hq * sp.n * D * sizeof(float) + 255) / 256) * 256)
                         : nullptr;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int G = Hq / Hkv;
  if (dtype == GQA_DTYPE_BF16) {
    if (!aligned(q, 16) || !aligned(kcache, 16) || !aligned(vcache, 16) || !aligned(out, 16))
      return GQA_ERR_INVALID_ARG;
    if ((D != 64 && D != 128) || G > 8) return GQA_ERR_UNSUPPORTED;
    if (B > 65535 || Hkv > 65535) return GQA_ERR_UNSUPPORTED;
    gqa::decode::Params p;
    p.q = static_cast<const __nv_bfloat16*>(q);
    p.kc = static_cast<const __nv_bfloat16*>(kcache);
    p.vc = static_cast<const __nv_bfloat16*>(vcache);
    p.seqlens = cache_seqlens;
    p.out = static_cast<__nv_bfloat16*>(out);
    p.part_o = part_o;
    p.part_lse = part_lse;
    p.B = B;
    p.Hq = Hq;
    p.Hkv = Hkv;
    p.G = G;
    p.Smax = max_seqlen_k;
    p.nsplit = sp.n;
    p.split_len = sp.len;
    p.scale_log2 = scale * kLog2e;
    const dim3 grid(sp.n, Hkv, B);
    if (!decode_smem_attr_set(current_device())) return GQA_ERR_CUDA;
    if (D == 64)
      gqa::decode::decode_split_kernel<64><<<grid, gqa::decode::kThreads, decode_smem_bytes<64>(), st>>>(p);
    else
      gqa::decode::decode_split_kernel<128><<<grid, gqa::decode::kThreads, decode_smem_bytes<128>(), st>>>(p);
    if (cudaGetLastError() != cudaSuccess) return GQA_ERR_CUDA;
    if (sp.n > 1) {
      __nv_bfloat16* ob = static_cast<__nv_bfloat16*>(out);
      const cudaError_t e =
          D == 128 ? launch_combine<__nv_bfloat16, 4>(st, part_o, part_lse, cache_seqlens, ob, B, Hq, D, sp.n, sp.len,
                                                      max_seqlen_k)
                   : launch_combine<__nv_bfloat16, 2>(st, part_o, part_lse, cache_seqlens, ob, B, Hq, D, sp.n, sp.len,
                                                      max_seqlen_k);
      if (e != cudaSuccess) return GQA_ERR_CUDA;
    }
    return GQA_OK;
  }
  if (dtype == GQA_DTYPE_FP32) {
    if (!aligned(q, 4) || !aligned(kcache, 4) || !aligned(vcache, 4) || !aligned(out, 4))
      return GQA_ERR_INVALID_ARG;
    if (D > gqa::f32::kMaxD) return GQA_ERR_UNSUPPORTED;
    gqa::f32::Params p{};
    p.q = static_cast<const float*>(q);
    p.k = static_cast<const float*>(kcache);
    p.v = static_cast<const float*>(vcache);
    p.out = static_cast<float*>(out);
    p.lse = nullptr;
    p.part_o = part_o;
    p.part_lse = part_lse;
    p.seqlens = cache_seqlens;
    p.q_sb = (long long)Hq * D;
    p.q_ss = 0;
    p.q_sh = D;
    p.k_sb = (long long)max_seqlen_k * Hkv * D;
    p.k_ss = (long long)Hkv * D;
    p.k_sh = D;
    p.B = B;
    p.Hq = Hq;
    p.Hkv = Hkv;
    p.G = G;
    p.Sq = 1;
    p.Sk = max_seqlen_k;
    p.D = D;
    p.causal = 0;
    p.scale = scale;
    p.nsplit = sp.n;
    p.split_len = sp.len;
    p.len_cap = max_seqlen_k;
    const int rc = launch_f32(p, st);
    if (rc != GQA_OK) return rc;
    if (sp.n > 1 && launch_combine<float, 1>(st, part_o, part_lse, cache_seqlens, static_cast<float*>(out), B, Hq, D,
                                             sp.n, sp.len, max_seqlen_k) != cudaSuccess)
      return GQA_ERR_CUDA;
    return GQA_OK;
  }
  return GQA_ERR_INVALID_ARG;
}

int gqa_bwd(const void* q, const void* k, const void* v, const void* out, const void* dout, const float* lse,
            float* dsum, void* dq, void* dk, void* dv, int B, int Hq, int Hkv, int Sq, int Sk, int D, float scale,
            int causal, const int* seqlens_k, int dtype, void* stream) {
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || Sq <= 0 || Sk <= 0 || D <= 0) return GQA_ERR_INVALID_ARG;
  if (Hq % Hkv != 0) return GQA_ERR_INVALID_ARG;
  if (!q || !k || !v || !out || !dout || !lse || !dsum || !dq || !dk || !dv) return GQA_ERR_INVALID_ARG;
  if (!std::isfinite(scale)) return GQA_ERR_INVALID_ARG;
  if (causal != 0 && causal != 1) return GQA_ERR_INVALID_ARG;
  if (!aligned(lse, 4) || !aligned(dsum, 4) || (seqlens_k && !aligned(seqlens_k, 4))) return GQA_ERR_INVALID_ARG;
  if (dtype != GQA_DTYPE_BF16) return dtype == GQA_DTYPE_FP32 ? GQA_ERR_UNSUPPORTED : GQA_ERR_INVALID_ARG;
  for (const void* t : {q, k, v, out, dout, static_cast<const void*>(dq), static_cast<const void*>(dk),
                        static_cast<const void*>(dv)})
    if (!aligned(t, 16)) return GQA_ERR_INVALID_ARG;
  if (D != 64 && D != 128) return GQA_ERR_UNSUPPORTED;
  if (Hq > 65535 || B > 65535 || (long long)Hq * D * Sq * B > (1LL << 40) ||
      (long long)Hkv * D * Sk * B > (1LL << 40))
    return GQA_ERR_UNSUPPORTED;
  if (Hq / Hkv > 128) return GQA_ERR_UNSUPPORTED;        // a 128-row tile holds one token of every head
  gqa::bwd::Params p{};
  p.o = static_cast<const __nv_bfloat16*>(out);
  p.dout = static_cast<const __nv_bfloat16*>(dout);
  p.lse = lse;
  p.seqlens = seqlens_k;
  p.dsum = dsum;
  p.dq = static_cast<__nv_bfloat16*>(dq);
  p.dk = static_cast<__nv_bfloat16*>(dk);
  p.dv = static_cast<__nv_bfloat16*>(dv);
  p.B = B;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.G = Hq / Hkv;
  p.Sq = Sq;
  p.Sk = Sk;
  p.causal = causal;
  p.scale = scale;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  return D == 64 ? launch_bwd<64>(p, q, k, v, st) : launch_bwd<128>(p, q, k, v, st);
}

int gqa_device_status(void* stream) {
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return GQA_ERR_CUDA;
  unsigned v = 0;
  if (cudaMemcpyFromSymbol(&v, gqa::g_error_word, sizeof(v)) != cudaSuccess) return GQA_ERR_CUDA;
  if (v != 0) {
    const unsigned zero = 0;
    if (cudaMemcpyToSymbol(gqa::g_error_word, &zero, sizeof(zero)) != cudaSuccess) return GQA_ERR_CUDA;
  }
  return int(v);
}

}  // extern "C"

// ===================================================== no-allocation decode
// A variant of gqa_decode for callers that cannot allocate device memory: the
// split partials live in a fixed scratch array that belongs to the library.
namespace {

// The size is the one gqa.h publishes (32 MiB per device).
constexpr size_t kStaticScratchBytes = size_t(GQA_DECODE_NOALLOC_SCRATCH_BYTES);
static_assert(kStaticScratchBytes == (size_t(32) << 20), "the header documents a 32 MiB scratch");

// File-scope device array: every device that loads this library holds one
// copy until the process exits.  In host code the name is only a stand-in
// for the symbol; the device address comes from cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_decode_scratch[kStaticScratchBytes];

std::mutex g_scratch_mu;
void* g_scratch_addr[kMaxDevices] = {nullptr};

// Device address of g_decode_scratch on device `dev` (which must be the
// current device), looked up once per device and cached.
void* static_scratch(int dev) {
  if (dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess) return nullptr;
    g_scratch_addr[dev] = p;
  }
  return g_scratch_addr[dev];
}

}  // namespace

extern "C" int gqa_decode_noalloc(const void* q, const void* kcache, const void* vcache,
                                  const int* cache_seqlens, void* out, int B, int Hq, int Hkv, int D,
                                  float scale, int num_splits, int max_seqlen_k, int dtype, void* stream) {
  const size_t need = gqa_decode_workspace_bytes(B, Hq, Hkv, D, num_splits, max_seqlen_k);
  if (need > kStaticScratchBytes) return GQA_ERR_UNSUPPORTED;
  void* ws = nullptr;
  if (need > 0) {
    ws = static_scratch(current_device());
    if (!ws) return GQA_ERR_CUDA;
  }
  // Nothing in the scratch has to start at zero: every split partial the
  // combine step reads is written earlier in the same call.
  return gqa_decode(q, kcache, vcache, cache_seqlens, out, B, Hq, Hkv, D, scale, num_splits, max_seqlen_k,
                    dtype, ws, need, stream);
}
