/*
 * apa.h -- C ABI of libapa.so: adaptive-precision causal attention prefill
 * with GQA packing on GB300 (sm_103a).
 *
 * The method is the one of "APA: sloppy attention, exact where it counts"
 * (rfriedmann.de blog):
 *   - pass 1 ("Pass 1: FP4 everywhere, with a hot test") computes every 64-key
 *     tile in block-scaled NVFP4 (E2M1 elements, one UE4M3 scale per 16 values,
 *     one FP32 scale per head; keys mean-centred per channel) and flags "hot"
 *     tiles, those where a row of a 16-row group has FP4 tile mass above
 *     eps times its running sum lambda;
 *   - pass 2 ("Pass 2: exact FP16 on the hot tiles") recomputes only the hot
 *     tiles exactly (here in BF16 with FP32 accumulation);
 *   - the two online-softmax states, which share one logit frame, are merged
 *     exactly by log-sum-exp ("The merge that makes it exact").
 * Shapes and masking follow SDPA (ffpa-attn.readthedocs.io, the "Note" on
 * cross-, GQA and causal attention): BHSD layout, Hq % Hkv == 0, and with
 * causal != 0 the queries are aligned to the key tail: query row i sees key j
 * iff j <= i + (Nkv - Nq), which needs Nkv >= Nq.  The softmax scale is 1/sqrt(d).
 *
 * Common conventions:
 *   - All pointer arguments of the device entry points are device memory owned
 *     by the caller; the library never frees them.  q, k, v must be 16-byte
 *     aligned.
 *   - Calls are asynchronous: they enqueue work on `stream` and return.
 *     Asynchronous kernel errors surface at the caller's next synchronisation;
 *     a device-side wait that timed out is recorded in a library-wide device
 *     error word that apa_check_error() reports.
 *   - Results are deterministic: reruns with the same inputs are bitwise equal.
 *   - On a negative status nothing has been enqueued.  No C++ exception crosses
 *     the ABI.
 */
#ifndef APA_H
#define APA_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

/* status codes */
#define APA_OK 0
#define APA_ERR_NULL (-1)      /* a required pointer is null */
#define APA_ERR_SHAPE (-2)     /* B, Hq, Hkv, Nq, Nkv out of range, Hq % Hkv != 0, or causal with Nkv < Nq */
#define APA_ERR_EPS (-3)       /* eps < 0 or NaN */
#define APA_ERR_HEAD_DIM (-4)  /* d not in {64, 128, 256} */
#define APA_ERR_CUDA (-5)      /* a CUDA call or launch failed; cudaGetLastError() holds the cause */
#define APA_ERR_NOMEM (-6)     /* the workspace could not be allocated, or the given one is too small */
#define APA_ERR_DEVICE (-7)    /* a kernel recorded a device-side error: a timeout, or a bad block-table entry (apa_check_error) */
#define APA_ERR_ALIGN (-8)     /* q, k or v not 16-byte aligned */
#define APA_ERR_SCRATCH (-9)   /* too large for the fixed scratch of apa_quantize_noalloc */
#define APA_ERR_FLAGS (-10)    /* an unknown bit in `flags` */

/* Options of the _ex entry points. */
#define APA_FLAG_Q_RESIDUAL 1u /* Q as two FP4 terms in pass 1 (see apa_attention_ex) */
#define APA_FLAG_LSE_SCALES 2u /* least-squared-error block scales for Q, K, V (see apa_attention_ex) */
#define APA_FLAG_VALUE_WEIGHTED 4u /* hot test weighted by value norm (see apa_attention_ex) */
#define APA_FLAG_ROWSUM_MMA 8u /* pass-1 tile row sums from an MMA against an E2M1 ones tile (see apa_attention_ex) */

/* Size of the fixed device scratch array behind apa_quantize_noalloc (16 MiB). */
#define APA_NOALLOC_SCRATCH_BYTES (16u * 1024u * 1024u)

/* Adaptive-precision attention, eps >= 0:
 *   q        bf16 [B, Hq, Nq, d], contiguous
 *   k, v     bf16 [B, Hkv, Nkv, d], contiguous
 *   causal   0: every key visible; else tail-aligned causal mask
 *   eps      hot-test threshold.  0 runs every visible tile exactly (the all-exact
 *            path: pass 2 only, Q K^T in BF16, P.V with P rounded once to FP16
 *            against an FP16 copy of V, FP32 accumulation); +inf makes every tile
 *            cold (all-FP4 pass 1).
 *   out      fp32 [B, Hq, Nq, d] (required)
 *   lse      fp32 [B, Hq, Nq], natural-log log-sum-exp of the scaled scores (nullable)
 *   hot_mask uint32 [B, Hkv, ceil(G*Nq/16), ceil(T/32)] with G = Hq/Hkv and
 *            T = ceil(Nkv/64): bit t%32 of word t/32 is set iff key tile t was
 *            hot for that 16-row group of GQA-packed rows (packed row p = pos*G + g
 *            holds query head h*G + g at position pos).  At eps = 0 every tile the
 *            group can see is marked.  Nullable.
 * The workspace is allocated stream-ordered on `stream` (cudaMallocAsync) and
 * released the same way.  Returns APA_OK or a negative status.
 * When the pass-1 CTAs leave at least 8 SMs free, the K/V tiles are quantized
 * inside the pass-1 launch ("What else is in the box" on the page: quantization
 * inside the launch): that kernel is then launched cooperatively with one block
 * on every SM, so it starts once the whole GPU is free and holds it while it
 * runs.  If the driver refuses that launch (fewer SMs available to the context
 * than the device has), the call falls back to the separate quantizer kernel.
 * The results are the same bits either way. */
int apa_attention(const void* q, const void* k, const void* v, int B, int Hq, int Hkv, int Nq, int Nkv, int d,
                  int causal, float eps, float* out, float* lse, uint32_t* hot_mask, cudaStream_t stream);

/* Bytes of device workspace apa_attention_ws() needs for this problem.  At
 * eps = 0 that is the FP16 copy of V ([B][Hkv][Nkv][d] FP16, V divided by a
 * power of two per head only when max |v| > 2^15, so exact for every bf16 value
 * above the FP16 subnormals) and the heads' maxima of |v|; at d = 256, when a KV
 * head has at most 4 blocks of 128 packed rows and 2048 or more key tiles, also
 * the (m, l, O) states of the parts into which each block's walk is split (one
 * part per 1024 tiles, at most 4).  At eps > 0 it holds the quantized operands,
 * the pass-1 states and the hot lists, and at d = 256, when a KV head has at most
 * 4 blocks and 1024 or more key tiles, the states of the parts of pass 2's walks
 * over the hot lists (one part per 512 tiles, at most 4). */
size_t apa_workspace_bytes(int B, int Hq, int Hkv, int Nq, int Nkv, int d, float eps);

/* apa_attention() with a caller-provided device workspace of at least
 * apa_workspace_bytes() bytes, 256-byte aligned; it allocates nothing.
 * Two calls that overlap on the GPU must not share a workspace. */
int apa_attention_ws(const void* q, const void* k, const void* v, int B, int Hq, int Hkv, int Nq, int Nkv, int d,
                     int causal, float eps, float* out, float* lse, uint32_t* hot_mask, void* workspace,
                     size_t workspace_bytes, cudaStream_t stream);

/* apa_attention() with options (APA_FLAG_*; unknown bits give APA_ERR_FLAGS):
 *   APA_FLAG_Q_RESIDUAL  Q goes to pass 1 as two FP4 terms ("Second hunt" on the
 *                        page): Q1 as before and Q2, the FP4 quantization of the
 *                        residual Q - Q1 under the same FP32 head scale (block
 *                        scales of its own; residual r = fp32(x - fp32(E2M1 *
 *                        UE4M3 * s)) per element).  Both terms accumulate into
 *                        the same S against the same K: twice the QK^T work of
 *                        pass 1, which then runs one 128-row block per CTA.
 *   APA_FLAG_LSE_SCALES  every block scale of Q, K, V (and of the residual Q
 *                        term) picked by least squared error instead of the
 *                        nearest one ("Second hunt"): among the nearest UE4M3
 *                        code and its two neighbours, tried in that order, the
 *                        one whose FP32 sum of squared errors over the 16 values
 *                        (in index order) is strictly smallest.
 *   APA_FLAG_VALUE_WEIGHTED  the hot test weighted by value norm ("Honest
 *                        limits" on the page: the plain test bounds a cold
 *                        tile's share of the softmax mass, not of the output):
 *                        tile t is hot iff some row has w_t * l_t > eps * lambda,
 *                        w_t = (largest key value norm in the tile) / (mean key
 *                        value norm of the head); norms are FP32 sums of FP32
 *                        squares in channel order with a rounded square root,
 *                        the mean follows the key mean's summation order.
 *                        lambda stays the plain running sum.  A cold tile then
 *                        moves each output row by at most eps times the mean
 *                        value norm.  Costs 8 bytes of workspace per tile.
 *   APA_FLAG_ROWSUM_MMA  the tile row sums l_t of pass 1 from one extra MMA of
 *                        the E2M1 P against an E2M1 ones tile ("Pass 1", step 3
 *                        on the page), instead of the default: each row's thread
 *                        sums its own E2M1 codes exactly in registers.  Both are
 *                        the exact sum of the quantized P; the MMA form runs one
 *                        128-row block per pass-1 CTA with the separate K/V
 *                        quantizer.  Not combinable with APA_FLAG_Q_RESIDUAL
 *                        (APA_ERR_FLAGS): both need the same TMEM columns.
 * `workspace` of at least apa_workspace_bytes_ex() bytes (256-byte aligned), or
 * null to have it allocated stream-ordered for the call. */
int apa_attention_ex(const void* q, const void* k, const void* v, int B, int Hq, int Hkv, int Nq, int Nkv, int d,
                     int causal, float eps, unsigned flags, float* out, float* lse, uint32_t* hot_mask,
                     void* workspace, size_t workspace_bytes, cudaStream_t stream);
size_t apa_workspace_bytes_ex(int B, int Hq, int Hkv, int Nq, int Nkv, int d, float eps, unsigned flags);

/* apa_attention() on a paged K/V cache.  Every (sequence, KV head) keeps its keys
 * and values in pages of 64 keys (one key tile) drawn from one pool:
 *   k_pages, v_pages  bf16 [num_pages][Hkv][64][d], contiguous, 16-byte aligned
 *   block_table       int32 [B][max_pages] in device memory: entry t of sequence b
 *                     is the page holding its keys 64t .. 64t+63;
 *                     max_pages >= ceil(Nkv/64); num_pages * Hkv * 64 < 2^31
 * (the blog, "What else is in the box": pass 2 reads through a block table; here
 * every read of K and V does).  All sequences have Nkv keys and Nq queries, as
 * in apa_attention.  Keys past Nkv in a sequence's last page are never used.  A
 * table entry outside [0, num_pages) reads page 0 and is reported by
 * apa_check_error as a bounds error (status APA_ERR_DEVICE).  The results are
 * those of apa_attention on the same keys laid out contiguously, bit for bit. */
int apa_attention_paged(const void* q, const void* k_pages, const void* v_pages, int num_pages,
                        const int32_t* block_table, int max_pages, int B, int Hq, int Hkv, int Nq, int Nkv, int d,
                        int causal, float eps, float* out, float* lse, uint32_t* hot_mask, cudaStream_t stream);

/* apa_attention() on HOST buffers (page-locked memory recommended): copies q, k,
 * v to the device, runs, copies out (and lse / hot_mask when non-null) back,
 * and synchronizes `stream` before returning.  The results equal those of
 * apa_attention().  Each (b, KV head) is an independent problem of the method,
 * so the call pipelines them: one's inputs are copied (on a library-owned copy
 * stream) while earlier ones compute (on up to 8 library-owned streams, created
 * at rising priority so that the sub-problems that arrive last are dispatched
 * first) and their results are copied back.  All of it is ordered after the work already
 * on `stream`.  The device memory is one library-owned buffer per device, grown
 * on demand and kept until the process exits; calls on the same device are
 * serialized by a lock. */
int apa_attention_host(const void* q, const void* k, const void* v, int B, int Hq, int Hkv, int Nq, int Nkv, int d,
                       int causal, float eps, float* out, float* lse, uint32_t* hot_mask, cudaStream_t stream);

/* Where, inside a caller's workspace, an eps > 0 call of apa_attention_ws() or
 * apa_attention_ex() (with these flags) leaves the pass-1 NVFP4 operands: byte
 * offsets of the K/V tile blobs, the Q blobs, the key mean and the FP32 head
 * scales, in the layouts apa_quantize() writes them.  They hold the call's
 * operands once the call has completed, until the workspace is used again; that
 * holds whether the K/V tiles were quantized by the separate kernel or inside
 * the pass-1 launch.  A measurement and testing aid, not needed to use the
 * library.  Returns APA_OK; APA_ERR_EPS for eps <= 0 (the all-exact path
 * quantizes nothing), or the argument errors of apa_attention_ex(). */
int apa_workspace_operands(int B, int Hq, int Hkv, int Nq, int Nkv, int d, float eps, unsigned flags,
                           size_t* kv_blob, size_t* q_blob, size_t* mu, size_t* s_q, size_t* s_k, size_t* s_v);

/* The pass-1 NVFP4 operands on their own (blog, "Pass 1" and "Mean-centred K"):
 *   kv_blob  uint8 [B*Hkv][T][apa_kv_blob_bytes / (B*Hkv*T)]: per 64-key tile the
 *            E2M1 codes of the centred keys and of V^T with their UE4M3 scales, in
 *            the tcgen05 shared-memory image (layout in the library's
 *            apa_internal.h; 9216 bytes per tile at d = 128)
 *   q_blob   uint8 [B*Hkv][ceil(G*Nq/128)][72*d]: E2M1 codes and UE4M3 scales of
 *            128 GQA-packed query rows per block
 *   mu       fp32 [B, Hkv, d]  per-channel key mean
 *   s_q      fp32 [B, Hq]; s_k, s_v fp32 [B, Hkv]: FP32 per-head scales
 * Temporary statistics are allocated stream-ordered on `stream`. */
int apa_quantize(const void* q, const void* k, const void* v, int B, int Hq, int Hkv, int Nq, int Nkv, int d,
                 uint8_t* kv_blob, uint8_t* q_blob, float* mu, float* s_q, float* s_k, float* s_v,
                 cudaStream_t stream);
size_t apa_kv_blob_bytes(int B, int Hkv, int Nkv, int d);
/* apa_quantize() with options: q2_blob (nullable, q_blob's layout) receives the
 * codes and scales of the FP4 residual term of Q (APA_FLAG_Q_RESIDUAL);
 * APA_FLAG_LSE_SCALES picks every block scale by least squared error.  The flag
 * APA_FLAG_Q_RESIDUAL is implied by a non-null q2_blob; APA_FLAG_VALUE_WEIGHTED
 * changes nothing here (the weights are not an operand). */
int apa_quantize_ex(const void* q, const void* k, const void* v, int B, int Hq, int Hkv, int Nq, int Nkv, int d,
                    unsigned flags, uint8_t* kv_blob, uint8_t* q_blob, uint8_t* q2_blob, float* mu, float* s_q,
                    float* s_k, float* s_v, cudaStream_t stream);

/* apa_quantize() for callers that must not allocate device memory during the
 * call: engines that reserve the whole GPU for their own memory arena up front,
 * plugin interfaces that receive buffers but have no allocator to call, and
 * latency-critical paths where a device allocation (which can synchronize) is
 * not acceptable.  The blog has no counterpart to this entry point.
 *   Same arguments, outputs and results as apa_quantize(); no cudaMalloc,
 *   cudaFree or other allocating call is made.  The temporary statistics live in
 *   one fixed array of APA_NOALLOC_SCRATCH_BYTES in the library's device image,
 *   which every GPU that loads the library holds until the process exits.
 *   Problems whose statistics need more than that
 *   (apa_quantize_noalloc_scratch_bytes() > APA_NOALLOC_SCRATCH_BYTES, roughly
 *   B*Hkv*ceil(Nkv/64)*d*4 bytes) are rejected with APA_ERR_SCRATCH before any
 *   work is enqueued.
 *   The first call on a device looks up the array's device address
 *   (cudaGetSymbolAddress) with that device current; make that first call before
 *   any stream capture.
 *   Every call shares the one array per device, and each call overwrites what
 *   the last one left there: calls that can overlap on the GPU (different
 *   streams without ordering between them) race on it and must be serialized by
 *   the caller. */
int apa_quantize_noalloc(const void* q, const void* k, const void* v, int B, int Hq, int Hkv, int Nq, int Nkv,
                         int d, uint8_t* kv_blob, uint8_t* q_blob, float* mu, float* s_q, float* s_k, float* s_v,
                         cudaStream_t stream);
/* Scratch bytes apa_quantize_noalloc needs for this problem (0 for invalid sizes). */
size_t apa_quantize_noalloc_scratch_bytes(int B, int Hq, int Hkv, int Nkv, int d);
size_t apa_q_blob_bytes(int B, int Hq, int Hkv, int Nq, int d);

/* Measurement aid, off by default.  While enabled, every apa_attention* call
 * records CUDA events on its stream around its three stages (quantizer, pass 1,
 * pass 2 with the merge); enabling or disabling resets the record. */
int apa_stage_timing(int enable);
/* Waits for the recorded events and returns the summed milliseconds per stage in
 * ms[0..2] (quantizer, pass 1, pass 2) and the number of calls in *calls, then
 * clears the record.  At eps = 0 only the pass-2 stage has work. */
int apa_stage_timing_read(float* ms, int* calls);

/* Synchronizes `stream`, then returns APA_ERR_DEVICE (and clears the word) if a
 * kernel of this library recorded a device-side timeout on the current device,
 * APA_ERR_CUDA if the stream reported an error, APA_OK otherwise. */
int apa_check_error(cudaStream_t stream);

/* Human-readable text for a status code (static storage). */
const char* apa_status_string(int status);

#ifdef __cplusplus
}
#endif
#endif /* APA_H */
