/*
 * gqa.h -- C ABI of libgqa, a grouped-query attention (GQA) forward library
 * for NVIDIA B300 (sm_103a).
 *
 * What it computes (sources cited by page title and section):
 *   [GQA-BERT]  "3个GQA核心优化技巧：解决BERT模型内存效率与吞吐量瓶颈"
 *               (blog.gitcode.com): "GQA的分组共享机制" -- Hq query heads are
 *               split into groups that share one K/V head, Hq % Hkv == 0,
 *               group size G = Hq / Hkv; "Flash-Attention的稀疏分组优化" --
 *               query head h reads K/V head h / G, and a K/V block staged in
 *               shared memory is reused by every query head of its group;
 *               "阶段二" -- softmax scale 1/sqrt(d_head), causal off for
 *               BERT, num_splits for split computation, seqlen_k hint.
 *   [GQA-PAPER] "GQA: Training Generalized Multi-Query Transformer Models
 *               from Multi-Head Checkpoints" (azimuth.plus/paper/gqa):
 *               "Idea 2" (GQA-H = MHA, GQA-1 = MQA, contiguous groups),
 *               "Problem"/"Bottleneck" (a decode step reads the whole KV
 *               cache; it is bandwidth bound), KV_cache_size equation.
 *   [LOWRANK]   aifullclass.xyz BERT attention article, code example:
 *               softmax(Q K^T * scale, masked keys excluded) V.
 *   [FA-SERIES] "FlashAttention Serisi: Bellek G/Ç Tıkanıklığının Çözümü"
 *               (webturing.pages.dev): "Ana fikir" (tiled online softmax,
 *               scores never written to slow memory, identical result),
 *               "V3 ve donanım uyumu" (warp-specialised producer/consumer).
 *
 *   For batch b, query head h (K/V head kvh = h / G), query row i:
 *     L_b = seqlens_k ? seqlens_k[b] : Sk          (right-padded keys)
 *     J   = { j < L_b  and  (!causal or j <= i + Sk - Sq) }
 *     out[b,i,h,:] = sum_{j in J} softmax_j(scale * q.k_j) v_j
 *     lse[b,h,i]   = ln sum_{j in J} exp(scale * q.k_j)
 *   An empty J gives out = 0 and lse = -inf.  Keys outside J get exactly
 *   zero weight (the page's -1e9 fill read as "never attended").
 *
 * Conventions shared by every entry point
 *   - All tensor pointers are DEVICE pointers owned by the caller; the
 *     library keeps no reference after the call returns and allocates no
 *     device memory per call.
 *   - Layouts are row-major and contiguous (BSHD, head dimension last):
 *       q, out [B, Sq, Hq, D];  k, v [B, Sk, Hkv, D];  lse [B, Hq, Sq] fp32
 *       decode: q, out [B, Hq, D];  kcache, vcache [B, Smax, Hkv, D]
 *   - dtype: GQA_DTYPE_BF16 (q/k/v/out bfloat16, fp32 accumulation,
 *     tcgen05 tensor cores) or GQA_DTYPE_FP32 (q/k/v/out float32, exact
 *     fp32 SIMT check path).  lse is always float32.
 *   - stream is a cudaStream_t (NULL = legacy default stream) of the
 *     CURRENT device, and every pointer lives on that device: the library
 *     reads the current device for its per-device state (SM count, kernel
 *     attributes, work-unit scheduler slots, scratch addresses).  Calls only
 *     enqueue work: they never synchronise, so errors found on the device
 *     (a key length out of range, a pipeline wait that timed out) are
 *     reported later by gqa_device_status().
 *   - Return value: a gqa_status code.  On any non-OK return nothing has
 *     been enqueued.
 *   - Bounded waits: every pipeline wait inside the prefill and backward
 *     kernels gives up after GQA_WAIT_TIMEOUT_NS nanoseconds (environment
 *     variable, default 2e9, read at each call); the CTA then drains its
 *     copies and matrix products, frees its tensor memory and exits, and the
 *     call reports GQA_ERR_DEVICE_TIMEOUT through gqa_device_status().
 *     Until that status has been read (which clears it), later launches on
 *     the device give up at their first wait that does not complete at once.
 *     A nonzero GQA_TEST_FORCE_TIMEOUT (read at each call) is a test hook:
 *     one MMA-issuing thread per CTA first waits on a barrier nothing
 *     arrives on, so that the abort path runs.
 */
#ifndef GQA_H_
#define GQA_H_

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    GQA_OK = 0,
    GQA_ERR_INVALID_ARG = 1,     /* bad size, pointer, alignment, Hq % Hkv != 0, ... */
    GQA_ERR_UNSUPPORTED = 2,     /* valid but not implemented (e.g. bf16 with D not 64/128) */
    GQA_ERR_CUDA = 3,            /* a CUDA runtime/driver call failed */
    GQA_ERR_DEVICE_TIMEOUT = 4,  /* a device-side pipeline wait gave up (reported by gqa_device_status) */
    GQA_ERR_DEVICE_BOUNDS = 5    /* a device-side length check failed (reported by gqa_device_status) */
} gqa_status;

/* Arithmetic path of a call.  The names carry a DTYPE_ infix (GQA_DTYPE_BF16
 * rather than GQA_BF16) so that they cannot be mistaken for status codes. */
typedef enum {
    GQA_DTYPE_BF16 = 0,
    GQA_DTYPE_FP32 = 1
} gqa_dtype;

/*
 * gqa_fwd -- prefill / encoder attention, non-causal (BERT) or causal.
 * [GQA-BERT] "GQA的分组共享机制", "Flash-Attention的稀疏分组优化", "阶段二";
 * [LOWRANK] code example; [FA-SERIES] "Ana fikir".
 *
 *   q         [B, Sq, Hq, D]   device, read
 *   k, v      [B, Sk, Hkv, D]  device, read
 *   out       [B, Sq, Hq, D]   device, written (same dtype as q)
 *   lse       [B, Hq, Sq] fp32 device, written; may be NULL (not written)
 *   B, Hq, Hkv, Sq, Sk, D      sizes, all >= 1; Hq % Hkv == 0 ([GQA-BERT])
 *   scale     finite softmax scale (the pages use 1/sqrt(D))
 *   causal    0: every query sees keys [0, L_b); 1: query row i also
 *             requires j <= i + Sk - Sq (bottom-right aligned)
 *   seqlens_k int32 [B] device, key lengths L_b in [0, Sk]; NULL = all Sk.
 *             Values outside [0, Sk] make the affected batch entry write
 *             zeros and raise GQA_ERR_DEVICE_BOUNDS in gqa_device_status().
 *   dtype     gqa_dtype
 *   stream    cudaStream_t
 * bf16: D must be 64 or 128 and G = Hq/Hkv <= 128; q/k/v/out 16-byte aligned.
 * fp32: 1 <= D <= 256; 4-byte aligned.
 * Concurrency (bf16): each call hands its work units out through one of 64
 * counter slots in device memory, taken round-robin per call; up to 64 calls
 * may be in flight on one device at once (on different streams), more must
 * be serialised by the caller.
 * Returns GQA_OK, GQA_ERR_INVALID_ARG, GQA_ERR_UNSUPPORTED or GQA_ERR_CUDA.
 */
int gqa_fwd(const void* q, const void* k, const void* v, void* out, float* lse,
            int B, int Hq, int Hkv, int Sq, int Sk, int D, float scale, int causal,
            const int* seqlens_k, int dtype, void* stream);

/*
 * gqa_fwd_host -- gqa_fwd for inputs and outputs that live in host memory:
 * the batch is cut into chunks of batch entries, and each chunk's inputs go
 * host -> device, its attention runs, and its outputs go device -> host, on
 * three streams so that the two copy directions and the computation of
 * different chunks overlap.  The computation is exactly gqa_fwd's (one
 * gqa_fwd launch per chunk on `stream`; the outputs equal gqa_fwd's bit for
 * bit).  [GQA-BERT] "阶段二" (a batch of encoder sequences); no page defines
 * the copy pipeline, which only moves the data the method reads and writes.
 *
 *   q_h, k_h, v_h     host, read; layouts as gqa_fwd.  For the copies to run
 *                     asynchronously and overlap, host buffers must be
 *                     page-locked (cudaHostAlloc / cudaHostRegister);
 *                     pageable memory still gives correct results, with
 *                     copies that do not overlap.
 *   out_h             host, written, [B, Sq, Hq, D]
 *   lse_h             host, written, [B, Hq, Sq] fp32; may be NULL
 *   seqlens_k_h       host int32 [B] or NULL, as gqa_fwd's seqlens_k
 *   q_d, k_d, v_d, out_d   device buffers of the full tensors' sizes, owned
 *                     by the caller (staging; the library allocates nothing)
 *   lse_d             device [B, Hq, Sq] fp32, or NULL when lse_h is NULL
 *   seqlens_d         device int32 [B], or NULL when seqlens_k_h is NULL
 *   chunk_b           batch entries per chunk; <= 0 = automatic (B / 8,
 *                     at least 1)
 *   other arguments   as gqa_fwd
 * The call returns after enqueueing; the host outputs are complete once
 * `stream` has completed (the library makes `stream` wait for its copy
 * streams).  The host input buffers must not change, and the host output
 * buffers must not be read, before that.  The copy streams and events are
 * created once per device, on the first call with that device current.
 * Each chunk is one gqa_fwd launch and counts towards gqa_fwd's limit of 64
 * launches in flight per device.
 * Returns GQA_OK, GQA_ERR_INVALID_ARG, GQA_ERR_UNSUPPORTED or GQA_ERR_CUDA.
 */
int gqa_fwd_host(const void* q_h, const void* k_h, const void* v_h, void* out_h, float* lse_h,
                 int B, int Hq, int Hkv, int Sq, int Sk, int D, float scale, int causal,
                 const int* seqlens_k_h, int dtype, void* q_d, void* k_d, void* v_d, void* out_d,
                 float* lse_d, int* seqlens_d, int chunk_b, void* stream);

/*
 * gqa_fwd_varlen -- gqa_fwd over sequences of different lengths packed
 * back to back without padding (the BERT batching case: [GQA-BERT]
 * "阶段二" passes padding_mask / seqlen_k for sequences of unequal length;
 * packing drops the padded query rows instead of computing and discarding
 * them).
 *
 *   q, out        [total_q, Hq, D]   device; rows cu_seqlens_q[b] ..
 *                                    cu_seqlens_q[b+1]-1 are sequence b
 *   k, v          [total_k, Hkv, D]  device; rows cu_seqlens_k[b] ..
 *   lse           [Hq, total_q] fp32 device, written; may be NULL
 *   cu_seqlens_q, cu_seqlens_k  int32 [B+1] device, cu[0] = 0, non-
 *                 decreasing, cu[B] <= total; Lq_b = cu_q[b+1]-cu_q[b] in
 *                 [0, max_seqlen_q], Lk_b likewise in [0, max_seqlen_k].
 *                 Values outside these ranges make the affected sequence
 *                 write nothing and raise GQA_ERR_DEVICE_BOUNDS in
 *                 gqa_device_status().
 *   B             number of sequences
 *   max_seqlen_q, max_seqlen_k  upper bounds of Lq_b / Lk_b (they size the
 *                 work grid, not the buffers)
 *   total_q, total_k  rows of the packed tensors (>= 1)
 *   causal        0, or 1: query i of sequence b sees keys
 *                 j <= i + Lk_b - Lq_b (bottom-right aligned per sequence)
 * For sequence b, query head h, query row i (0 <= i < Lq_b) the result is
 * gqa_fwd's definition with L_b = Lk_b, Sq = Lq_b, Sk = Lk_b; rows of the
 * packed output that belong to no sequence are not written.
 * bf16: D 64 or 128, G <= 128, q/k/v/out 16-byte aligned.  fp32: D <= 256.
 * Concurrency as gqa_fwd.
 */
int gqa_fwd_varlen(const void* q, const void* k, const void* v, void* out, float* lse,
                   const int* cu_seqlens_q, const int* cu_seqlens_k, int B, int Hq, int Hkv,
                   int max_seqlen_q, int max_seqlen_k, int total_q, int total_k, int D,
                   float scale, int causal, int dtype, void* stream);

/*
 * gqa_fwd_sparse -- gqa_fwd restricted by a block-sparsity mask ([GQA-BERT]
 * "阶段二": block_size and sparse=True; the pages do not state the pattern,
 * so it is the caller's).  Key blocks that no query of a work unit keeps are
 * skipped (never loaded, never multiplied).
 *
 *   block_mask  uint8 [ceil(Sq/bs), ceil(Sk/bs)] device, row-major; nonzero
 *               = the queries of block i // bs may attend to the keys of
 *               block j // bs.  Shared by every batch entry and head.
 *   block_size  bs, 64 or 128 (GQA_ERR_INVALID_ARG otherwise)
 *   everything else as gqa_fwd (dense layout, seqlens_k, causal, lse).
 * Key j is admissible for query i when j < L_b, the causal condition holds
 * (if causal) and block_mask[i/bs][j/bs] != 0; rows with no admissible key
 * give out = 0 and lse = -inf.  bf16: Sk <= 8192 (GQA_ERR_UNSUPPORTED
 * otherwise), D 64 or 128, G <= 128.  fp32: as gqa_fwd.
 */
int gqa_fwd_sparse(const void* q, const void* k, const void* v, void* out, float* lse,
                   const unsigned char* block_mask, int block_size, int B, int Hq, int Hkv,
                   int Sq, int Sk, int D, float scale, int causal, const int* seqlens_k,
                   int dtype, void* stream);

/*
 * gqa_bwd -- gradients of gqa_fwd (dense layout) with respect to q, k and v
 * for an upstream gradient dout ([FA-SERIES] "V2 katkısı" names a faster backward
 * pass as one of its gains, and "Ana fikir" keeps the softmax intermediates
 * out of slow memory; read here as: the weights are rebuilt from the
 * forward's log-sum-exp, never stored.  [GQA-BERT] "GQA的分组共享机制": the
 * G query heads of a group read one K/V head, so that head's gradient sums
 * over the group).  With P_ij = exp(scale q_i.k_j - lse_i) over
 * the admissible keys of gqa_fwd and Dsum_i = dout_i . out_i:
 *     dv_j = sum_{h in group} sum_i P_ij dout_i
 *     dS_ij = P_ij (dout_i . v_j - Dsum_i)
 *     dq_i = scale sum_j dS_ij k_j
 *     dk_j = scale sum_{h in group} sum_i dS_ij q_i
 *
 *   q, out, dout  [B, Sq, Hq, D] bf16 device (out: the forward's output)
 *   k, v          [B, Sk, Hkv, D] bf16 device
 *   lse           [B, Hq, Sq] fp32 device: the forward's log-sum-exp (rows
 *                 with no admissible key hold -inf)
 *   dsum          [B, Hq, Sq] fp32 device, caller-owned scratch; written
 *                 with Dsum_i
 *   dq            [B, Sq, Hq, D] bf16 device, written (every element)
 *   dk, dv        [B, Sk, Hkv, D] bf16 device, written (every element;
 *                 keys >= L_b get zeros)
 *   scale, causal, seqlens_k  as gqa_fwd (and must be what it was given)
 *   dtype         GQA_DTYPE_BF16 only (GQA_DTYPE_FP32 -> GQA_ERR_UNSUPPORTED)
 * D 64 or 128, G = Hq/Hkv <= 128, B and Hq <= 65535 (GQA_ERR_UNSUPPORTED
 * otherwise); all bf16 tensors 16-byte aligned, lse and dsum 4-byte aligned
 * (GQA_ERR_INVALID_ARG otherwise, as for a NULL pointer, Hq % Hkv != 0, a
 * non-finite scale or causal not 0/1).  A key length outside [0, Sk] raises
 * GQA_ERR_DEVICE_BOUNDS in gqa_device_status() and counts as 0; a wait that
 * gives up raises GQA_ERR_DEVICE_TIMEOUT.  Gradients accumulate in fp32; P
 * and dS are rounded to bf16 for the products.  No atomics: the result does
 * not depend on scheduling.  Buffers must not overlap.  Launches three
 * kernels and returns without synchronising: Dsum and dK/dV on `stream`, dQ
 * on a side stream the library keeps per device, forked from `stream` after
 * Dsum and joined back to it by events, so every output is ready in
 * `stream` order (and a stream capture records both branches).
 */
int gqa_bwd(const void* q, const void* k, const void* v, const void* out, const void* dout,
            const float* lse, float* dsum, void* dq, void* dk, void* dv, int B, int Hq, int Hkv,
            int Sq, int Sk, int D, float scale, int causal, const int* seqlens_k, int dtype,
            void* stream);

/*
 * gqa_decode_num_splits -- the number of KV-length splits gqa_decode will use.
 * num_splits in 1..128 is returned clamped to the number of 16-key blocks of
 * max_seqlen_k; num_splits <= 0 asks for the automatic choice, which sizes
 * the grid to fill the GPU of the current device; num_splits > 128 is
 * rejected (-GQA_ERR_INVALID_ARG).
 * Split s of every sequence covers keys [s*Ls, (s+1)*Ls) with
 * Ls = ceil(max_seqlen_k / n) rounded up to 16 ([GQA-BERT] "阶段二":
 * num_splits cuts the key range into pieces computed independently).
 * Returns n >= 1, or a negative gqa_status on bad arguments.
 */
int gqa_decode_num_splits(int B, int Hkv, int max_seqlen_k, int num_splits);

/*
 * gqa_decode_workspace_bytes -- device scratch gqa_decode needs for the
 * split partials: fp32 O_s [B, Hq, n, D] plus fp32 lse_s [B, Hq, n], where
 * n = gqa_decode_num_splits(B, Hkv, max_seqlen_k, num_splits).  Returns 0
 * when n == 1 (no combine step) and 0 for invalid arguments.  Hkv is an
 * argument because the automatic split count (num_splits <= 0) depends on
 * the number of (batch, K/V head) pairs the split kernel runs over.  No page
 * defines this call: it sizes the caller-owned workspace of the split step.
 */
size_t gqa_decode_workspace_bytes(int B, int Hq, int Hkv, int D, int num_splits,
                                  int max_seqlen_k);

/*
 * gqa_decode -- one generated token per sequence attending to its KV cache.
 * [GQA-PAPER] "Problem"/"Bottleneck" (every step reads the whole cache);
 * [GQA-BERT] "阶段二" (num_splits); [FA-SERIES] "Ana fikir" (split partial
 * softmax results merge exactly through their log-sum-exp).
 *
 *   q              [B, Hq, D]          device, read
 *   kcache, vcache [B, Smax, Hkv, D]   device, read; Smax = max_seqlen_k
 *   cache_seqlens  int32 [B]           device; L_b in [0, Smax].  Out-of-range
 *                  values write zeros for that entry and raise
 *                  GQA_ERR_DEVICE_BOUNDS in gqa_device_status().
 *   out            [B, Hq, D]          device, written
 *   B, Hq, Hkv, D  sizes; Hq % Hkv == 0
 *   scale          finite softmax scale
 *   num_splits     <= 0 automatic, else 1..128 (see gqa_decode_num_splits)
 *   max_seqlen_k   Smax, the cache capacity (row stride of the caches)
 *   dtype          gqa_dtype
 *   workspace      device scratch of at least gqa_decode_workspace_bytes()
 *                  bytes, 16-byte aligned; may be NULL when that is 0.
 *                  Caller-owned; must not be used by another call in flight.
 *   workspace_bytes its size
 *   stream         cudaStream_t
 * bf16: D must be 64 or 128 and G <= 8 (GQA_ERR_UNSUPPORTED otherwise).
 * fp32: 1 <= D <= 256.  The new token sees the whole cached prefix (no
 * causal term).
 */
int gqa_decode(const void* q, const void* kcache, const void* vcache,
               const int* cache_seqlens, void* out, int B, int Hq, int Hkv, int D,
               float scale, int num_splits, int max_seqlen_k, int dtype,
               void* workspace, size_t workspace_bytes, void* stream);

/*
 * gqa_decode_fp8 -- gqa_decode over a KV cache stored as FP8 e4m3 (one byte
 * per value), half the bytes of a bf16 cache.  [GQA-PAPER] "Problem" /
 * "Bottleneck" (the step reads the whole cache, so its size sets the time);
 * [GQA-BERT] names quantisation of the cache as further compression.
 *
 *   q              [B, Hq, 128] bf16   device, read
 *   kcache, vcache [B, Smax, Hkv, 128] e4m3 (OCP FP8 E4M3, finite values
 *                  only, max 448) device, read
 *   k_scale, v_scale  one scale per tensor: the cached key is
 *                  k_scale * kcache and the value v_scale * vcache (the
 *                  caller quantises x as round(x / scale) to e4m3)
 *   everything else as gqa_decode (bf16 out, cache_seqlens, scale,
 *   num_splits, max_seqlen_k), except that the split count is
 *   gqa_decode_fp8_num_splits(...) and the workspace needs
 *   gqa_decode_fp8_workspace_bytes(B, Hq, Hkv, 128, num_splits,
 *   max_seqlen_k) bytes.
 * Result: gqa_decode's definition on the dequantised cache.  D must be 128
 * and G <= 8 (GQA_ERR_UNSUPPORTED otherwise); q/out/caches 16-byte aligned;
 * scale, k_scale and v_scale finite (GQA_ERR_INVALID_ARG otherwise).
 */
int gqa_decode_fp8(const void* q, const void* kcache, const void* vcache,
                   const int* cache_seqlens, void* out, int B, int Hq, int Hkv, int D,
                   float scale, float k_scale, float v_scale, int num_splits, int max_seqlen_k,
                   void* workspace, size_t workspace_bytes, void* stream);

/*
 * gqa_decode_fp8_num_splits / gqa_decode_fp8_workspace_bytes -- the split
 * count and workspace size of gqa_decode_fp8, with the same arguments,
 * clamping, return values and errors as gqa_decode_num_splits /
 * gqa_decode_workspace_bytes.  Only the automatic choice (num_splits <= 0)
 * differs: about 512 keys per split instead of 1024, because each FP8 CTA
 * streams four K/V heads at half the bytes per key.  No page defines these
 * calls: they size the caller-owned workspace of the FP8 split step.
 */
int gqa_decode_fp8_num_splits(int B, int Hkv, int max_seqlen_k, int num_splits);
size_t gqa_decode_fp8_workspace_bytes(int B, int Hq, int Hkv, int D, int num_splits,
                                      int max_seqlen_k);

/*
 * gqa_decode_noalloc -- gqa_decode for callers that cannot allocate device
 * memory.  The pages have no counterpart to this entry point.
 *
 * Some callers only ever receive the input and output buffers -- an operator
 * or plugin interface of a host framework that owns all device memory -- and
 * others must not allocate on the decode path at all, because cudaMalloc can
 * synchronise the device and takes unbounded time.  Those callers cannot
 * provide gqa_decode's split workspace.  This entry point takes the same
 * arguments as gqa_decode minus the workspace and puts the split partials in
 * a scratch array of GQA_DECODE_NOALLOC_SCRATCH_BYTES (32 MiB) that the
 * library holds in device memory: one file-scope device array per device that
 * loads the library, kept until the process exits.  No call allocates or
 * frees anything.
 *
 *   - Size limit: calls whose split partials would need more than 32 MiB
 *     (gqa_decode_workspace_bytes(B, Hq, Hkv, D, num_splits, max_seqlen_k)
 *     > GQA_DECODE_NOALLOC_SCRATCH_BYTES) return GQA_ERR_UNSUPPORTED and
 *     enqueue nothing; lower num_splits or use gqa_decode.
 *   - Set-up: the first call on a device looks up the scratch array's
 *     device address (once per device, with that device current).  Make that
 *     first call before any stream capture on the device.
 *   - Sharing: every call on a device uses the same scratch array, which
 *     keeps the previous call's contents (nothing in it has to start at zero).
 *     Calls that overlap on the GPU -- on different streams, or from several
 *     host threads -- race on it; serialise them.
 *   - Everything else (arguments, layouts, errors) is as for gqa_decode.
 */
#define GQA_DECODE_NOALLOC_SCRATCH_BYTES (32u << 20)
int gqa_decode_noalloc(const void* q, const void* kcache, const void* vcache,
                       const int* cache_seqlens, void* out, int B, int Hq, int Hkv, int D,
                       float scale, int num_splits, int max_seqlen_k, int dtype, void* stream);

/*
 * gqa_device_status -- synchronises `stream`, then returns and clears the
 * library's device error word for the current device: GQA_OK,
 * GQA_ERR_DEVICE_BOUNDS or GQA_ERR_DEVICE_TIMEOUT (GQA_ERR_CUDA if the
 * synchronisation itself failed).  The stream's device must be the current
 * device.  No page defines this call: it reports the device-side checks of
 * the kernels (key lengths, bounded pipeline waits).
 */
int gqa_device_status(void* stream);

/* gqa_status_string -- static, human-readable name of a status code.  No
 * page defines this call. */
const char* gqa_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* GQA_H_ */
