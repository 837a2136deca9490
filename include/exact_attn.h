/*
 * exact_attn.h — C ABI of the GB300 (sm_103a) exact-attention library.
 *
 * The library computes exact scaled-dot-product attention,
 *     O = softmax(scale * Q K^T + causal mask) V,
 * as defined in "Why Fast GPUs Still Wait for Memory"
 * (srini-anirudh.github.io), section "Attention from first principles"
 * (S = QK^T, P = softmax(S), O = PV), computed the IO-aware way described in
 * the section "FlashAttention is an IO algorithm" on the same page: K/V blocks
 * stream through on-chip memory and a running maximum and normaliser rescale
 * the output block, so the n x n score matrix never reaches HBM.  Causal
 * masking follows that page's note "causal masking is not an optimisation
 * here"; single-token decode follows its section "Attention III · KV cache,
 * GQA, MLA"; split-KV decode with a partial-output reduction follows the
 * schedule table of "M4.2 GPU Execution Model" (numinens.com), section 0x08
 * ("split-K ... partial-output reduction, workspace") and its prefill/decode
 * example in the operation atlas.
 *
 * Conventions shared by every entry point
 *   - All tensor pointers are DEVICE pointers owned by the caller; the library
 *     never frees them and keeps no reference after the call returns.
 *   - bf16 tensors are contiguous, row-major, head dimension innermost
 *     ([B, H, N, d] for the forward, [B, H, L, d] for the caches), and must be
 *     16-byte aligned.  d must be 64 or 128.
 *   - Work is enqueued on `stream` and runs asynchronously: the call returns
 *     after the launch without synchronising.  A NULL stream is the legacy
 *     default stream.
 *   - Arguments are validated on the host before anything is launched; an
 *     invalid call returns an error code and launches nothing.
 *   - Launch failures return ATTN_ERR_CUDA.  A device-side wait that exceeds
 *     its bounded limit records ATTN_ERR_TIMEOUT in a device status word that
 *     attn_get_device_status() reads and clears; the kernel then skips its
 *     remaining work and exits cleanly instead of hanging.
 *   - Every entry point may be called from several host threads.
 */
#ifndef EXACT_ATTN_H
#define EXACT_ATTN_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    ATTN_OK = 0,
    ATTN_ERR_NULL = 1,     /* a required pointer is NULL                        */
    ATTN_ERR_SHAPE = 2,    /* B, H, N or L out of range (< 1 or too large)      */
    ATTN_ERR_HEADDIM = 3,  /* d is not 64 or 128                                */
    ATTN_ERR_ALIGN = 4,    /* a tensor pointer is not 16-byte aligned           */
    ATTN_ERR_CUDA = 5,     /* a CUDA runtime/driver call or launch failed       */
    ATTN_ERR_NOMEM = 6,    /* workspace allocation failed / too small           */
    ATTN_ERR_TIMEOUT = 7,  /* a bounded device-side wait expired                */
    ATTN_ERR_ARG = 8       /* another argument is invalid (scale, causal flag),
                              or a kernel met an invalid index (a page id)      */
} attn_status;

/*
 * attn_fwd — fused forward attention for B*H independent heads.
 *
 *   Q, K, V : bf16 [B, H, N, d], contiguous.
 *   O       : bf16 [B, H, N, d] output, contiguous; O = P V / rowsum(P).
 *   LSE     : fp32 [B, H, N] output; LSE[i] = ln sum_j exp(scale * q_i . k_j)
 *             over the keys visible to query i (natural log, scale included).
 *   N       : sequence length, 1 <= N <= 2^24 (queries and keys alike).
 *   scale   : multiplies Q K^T before masking and softmax (finite, > 0).
 *   causal  : 0 = every key visible; 1 = key j visible to query i iff j <= i.
 *
 * One tcgen05/TMA kernel launch on a persistent grid of min(#SMs, work
 * items) CTAs, one per SM.  A work item is 256 query rows (two 128-row tiles)
 * of one head; each CTA starts with one item and claims the next from a
 * per-launch counter in a library-owned device array once it has issued the
 * current item's loads (causal: longest items first).  No workspace; S and P
 * stay on chip.  O and LSE are written exactly once per element.  O must not
 * alias Q, K or V.
 */
attn_status attn_fwd(const void *Q, const void *K, const void *V, void *O, float *LSE,
                     int B, int H, int N, int d, float scale, int causal,
                     cudaStream_t stream);

/*
 * attn_decode — one query token per (batch, head) against a KV cache.
 *
 *   q       : bf16 [B, H, d].
 *   Kcache  : bf16 [B, H, L, d];  Vcache : bf16 [B, H, L, d].
 *   O       : bf16 [B, H, d] output.
 *   L       : cache length, 1 <= L <= 2^24.  The new token follows the cache,
 *             so all L keys are visible (no mask).
 *
 * Split-KV: each head's keys are cut into s chunks of ceil(L/s) keys, s a
 * power of two chosen from the shape: the one nearest (in ratio) to 108 split
 * CTAs per SM over the call, i.e. 108 * SMs / (B*H) per head, raised to at
 * least 4 and capped at 32, then halved while a chunk would hold fewer than 64
 * keys (B=16, H=32, L=8192 on 152 SMs: s = 32; B=64, H=32, L=2048: s = 8).
 * One launch computes every chunk's normalised partial output and log-sum-exp
 * into a workspace (sized for 32 chunks whatever s is), a second launch
 * combines them with weights exp(lse_s - max_s lse_s).  The workspace is owned by the library: it is
 * allocated on first use per device, grows when a larger call needs it and
 * lives until process exit.  Growing it synchronises the device, so warm it up
 * with the largest shape before capturing a CUDA graph.  Calls that share a
 * device share that workspace, so concurrent calls on different streams of
 * one device race; use attn_decode_ws with separate workspaces for that.
 */
attn_status attn_decode(const void *q, const void *Kcache, const void *Vcache, void *O,
                        int B, int H, int L, int d, float scale, cudaStream_t stream);

/* Bytes of workspace attn_decode_ws needs for this shape (0 if invalid). */
size_t attn_decode_workspace_bytes(int B, int H, int L, int d);

/*
 * attn_decode_ws — attn_decode with a caller-owned device workspace of at
 * least attn_decode_workspace_bytes(B, H, L, d) bytes, 16-byte aligned.
 * Returns ATTN_ERR_NOMEM if ws_bytes is too small.  The workspace holds fp32
 * partials only while the call's two launches run; the caller may reuse it
 * for another call on the same stream afterwards.
 */
attn_status attn_decode_ws(const void *q, const void *Kcache, const void *Vcache, void *O,
                           int B, int H, int L, int d, float scale, void *ws,
                           size_t ws_bytes, cudaStream_t stream);

/*
 * Grouped-query attention ("Why Fast GPUs Still Wait for Memory", section
 * "Attention III · KV cache, GQA, MLA": h query heads share h_kv key/value
 * heads, group size g = h / h_kv, MQA being g = h; "M4.2 GPU Execution Model
 * for Transformer Kernels", example "logical GQA savings require a physical
 * grouped path").  Query head h of a batch reads K/V head floor(h / g)
 * (contiguous groups).  The K/V tensors keep their H_kv heads: nothing is
 * expanded, and each K/V tile is loaded once per group (the decode) or shared
 * through L2 by the group's neighbouring CTAs (the forward).
 *
 * attn_fwd_gqa — attn_fwd with Q, O bf16 [B, H, N, d], LSE fp32 [B, H, N] and
 * K, V bf16 [B, H_kv, N, d].  1 <= H_kv, H % H_kv == 0 (else ATTN_ERR_SHAPE);
 * H_kv == H is attn_fwd.  Everything else as attn_fwd.
 */
attn_status attn_fwd_gqa(const void *Q, const void *K, const void *V, void *O, float *LSE,
                         int B, int H, int H_kv, int N, int d, float scale, int causal,
                         cudaStream_t stream);

/*
 * attn_decode_gqa — attn_decode with q, O bf16 [B, H, d] and Kcache, Vcache
 * bf16 [B, H_kv, L, d].  One CTA per (batch, K/V head, up to 16 query heads of
 * its group, split) streams its K/V chunk once for all of those query heads,
 * which form the rows of tensor-core products against each K/V tile.
 * Uses the library-owned workspace of attn_decode (same size rule, same
 * stream caveats); H_kv == H is attn_decode.
 * attn_decode_gqa_ws — the same with a caller-owned workspace of at least
 * attn_decode_workspace_bytes(B, H, L, d) bytes (per query head).
 */
attn_status attn_decode_gqa(const void *q, const void *Kcache, const void *Vcache, void *O,
                            int B, int H, int H_kv, int L, int d, float scale,
                            cudaStream_t stream);
attn_status attn_decode_gqa_ws(const void *q, const void *Kcache, const void *Vcache, void *O,
                               int B, int H, int H_kv, int L, int d, float scale, void *ws,
                               size_t ws_bytes, cudaStream_t stream);

/*
 * attn_decode_paged — decode against a paged KV cache ("M4.2 GPU Execution
 * Model for Transformer Kernels": logical K/V continuity does not imply
 * contiguous physical addresses; the kernel contract includes the page/block
 * layout; pitfall 16 of the same page).
 *
 *   q, O        : bf16 [B, H, d].
 *   K_pages,
 *   V_pages     : bf16 [num_pages, H_kv, page_size, d] (one page holds
 *                 page_size consecutive tokens of every K/V head).
 *   block_table : int32 [B, max_blocks], device memory: token t of sequence b
 *                 is in page block_table[b * max_blocks + t / page_size],
 *                 slot t % page_size.
 *   seq_lens    : int32 [B], device memory: tokens of each sequence (clamped
 *                 to [0, max_blocks * page_size]; a sequence with no tokens
 *                 gets O = 0).
 *   page_size   : power of two, 1..65536; max_blocks * page_size <= 2^24.
 *   H_kv        : K/V heads (grouped-query attention as in attn_decode_gqa;
 *                 H_kv == H for multi-head).
 *
 * All sequences attend to all of their tokens (no mask).  Same split-KV
 * scheme, library-owned workspace and stream caveats as attn_decode.  A page
 * id outside [0, num_pages) is never dereferenced: the kernel skips those
 * tokens and records the error, which the next attn_get_device_status call
 * reports as ATTN_ERR_ARG (the outputs of that call are then not meaningful).
 */
attn_status attn_decode_paged(const void *q, const void *K_pages, const void *V_pages,
                              const int *block_table, const int *seq_lens, void *O, int B, int H,
                              int H_kv, int num_pages, int page_size, int max_blocks, int d,
                              float scale, cudaStream_t stream);

/*
 * attn_fwd_fp8 — attn_fwd with 8-bit floating-point (E4M3) Q, K and V ("Why
 * Fast GPUs Still Wait for Memory": the FP8 tensor ceiling is twice the bf16
 * one, roofline ceiling table).  Each input is E4M3 codes [B, H, N, d] with
 * one descale factor per tensor (value = code * descale, descale finite > 0);
 * the scores, the softmax and the accumulators are fp32, P is rounded to E4M3
 * (as P * 2^6, with every P <= 4) for the P V product.
 *
 *   Q8, K8, V8 : E4M3 [B, H, N, d], contiguous, 16-byte aligned; d == 128
 *                (else ATTN_ERR_HEADDIM).
 *   O          : bf16 [B, H, N, d];  LSE : fp32 [B, H, N] (natural log, with
 *                scale and descales applied), 4-byte aligned.
 *   scale      : multiplies the dequantised Q K^T, as in attn_fwd.
 *
 * Two launches on `stream`: a pass that writes V^T (d x N bytes per head)
 * into the workspace, and the persistent forward kernel of attn_fwd (items of
 * 256 query rows of one head, one CTA per SM).  attn_fwd_fp8 uses a library-owned grow-only workspace (its
 * own, same caveats as attn_decode); attn_fwd_fp8_ws takes a caller-owned one
 * of at least attn_fwd_fp8_workspace_bytes(B, H, N, d) bytes (ATTN_ERR_NOMEM
 * if smaller; 0 bytes is returned for an invalid shape).
 */
attn_status attn_fwd_fp8(const void *Q8, const void *K8, const void *V8, void *O, float *LSE,
                         int B, int H, int N, int d, float scale, float descale_q,
                         float descale_k, float descale_v, int causal, cudaStream_t stream);
attn_status attn_fwd_fp8_ws(const void *Q8, const void *K8, const void *V8, void *O, float *LSE,
                            int B, int H, int N, int d, float scale, float descale_q,
                            float descale_k, float descale_v, int causal, void *ws,
                            size_t ws_bytes, cudaStream_t stream);
size_t attn_fwd_fp8_workspace_bytes(int B, int H, int N, int d);

/*
 * attn_bwd — gradients of attn_fwd with respect to Q, K and V ("Why Fast GPUs
 * Still Wait for Memory", section "FlashAttention is an IO algorithm": the
 * backward pass keeps the tiling and recomputes S from Q and K instead of
 * storing it).  With the forward's output O and log-sum-exp LSE:
 *     P  = exp(scale Q K^T - LSE)      (causal mask as attn_fwd)
 *     dV = P^T dO,   dP = dO V^T,   dS = P * (dP - rowsum(dO * O))
 *     dQ = scale dS K,   dK = scale dS^T Q
 *
 *   Q, O, dO, dQ : bf16 [B, H, N, d], contiguous, 16-byte aligned.
 *   K, V, dK, dV : bf16 [B, H, N, d] (attn_bwd_gqa: [B, H_kv, N, d]).
 *   LSE          : fp32 [B, H, N], natural log, as attn_fwd wrote it
 *                  (4-byte aligned).
 *   scale, causal: those of the forward call.
 *
 * dQ, dK and dV are overwritten (never accumulated into) and must not overlap
 * any input.  Three launches on `stream`: a row pass (-rowsum(dO * O) and -LSE
 * in base 2 into the workspace), a dK/dV kernel (items: K/V head and 128-key
 * tile) and a dQ kernel (items: query head and 128-query tile), each on a
 * persistent grid of one CTA per SM that claims its items from a per-launch
 * counter.
 * No atomics: results are identical from run to run.  The workspace
 * (attn_bwd_workspace_bytes) is library-owned and grow-only as for
 * attn_decode, with the same synchronisation and stream caveats; it is not
 * shared with the decode workspace.  Validation and errors as attn_fwd.
 */
attn_status attn_bwd(const void *Q, const void *K, const void *V, const void *O, const void *dO,
                     const float *LSE, void *dQ, void *dK, void *dV, int B, int H, int N, int d,
                     float scale, int causal, cudaStream_t stream);

/*
 * attn_bwd_gqa — attn_bwd with H_kv K/V heads (1 <= H_kv, H % H_kv == 0, else
 * ATTN_ERR_SHAPE): K, V, dK, dV are [B, H_kv, N, d] and the gradient of a
 * K/V head sums those of the g = H / H_kv query heads that read it.
 * attn_bwd_gqa_ws — the same with a caller-owned workspace of at least
 * attn_bwd_workspace_bytes(B, H, N, d) bytes, 16-byte aligned (ATTN_ERR_NOMEM
 * if smaller); it is only used while the call's launches run.
 */
attn_status attn_bwd_gqa(const void *Q, const void *K, const void *V, const void *O,
                         const void *dO, const float *LSE, void *dQ, void *dK, void *dV, int B,
                         int H, int H_kv, int N, int d, float scale, int causal,
                         cudaStream_t stream);
attn_status attn_bwd_gqa_ws(const void *Q, const void *K, const void *V, const void *O,
                            const void *dO, const float *LSE, void *dQ, void *dK, void *dV, int B,
                            int H, int H_kv, int N, int d, float scale, int causal, void *ws,
                            size_t ws_bytes, cudaStream_t stream);

/* Bytes of workspace the backward needs: 2 * B * H * ceil(N/128) * 128 * 4
 * (0 if the shape is invalid). */
size_t attn_bwd_workspace_bytes(int B, int H, int N, int d);

/*
 * attn_decode_noalloc — attn_decode for callers that cannot allocate device
 * memory.  (The pages describe no such entry point; it has no counterpart
 * there.)
 *
 * Some callers can't let a library call cudaMalloc: a serving process whose
 * own allocator has already reserved nearly all of the GPU's memory, code that
 * must not have cudaMalloc/cudaFree block or synchronise the device in the
 * middle of its work, or a host framework that forbids plug-ins from
 * allocating device memory themselves.  This call computes the same result as
 * attn_decode with the same kernels, but its partials live in a fixed scratch
 * array compiled into the library: 16 MiB of device memory that every GPU
 * which loads the library holds until the process exits.  It never calls
 * cudaMalloc, cudaFree or any allocating routine.  The caller still passes
 * q, the caches and O.
 *
 *   Limit: B*H*32*(d+1)*4 bytes of partials must fit in 16 MiB
 *          (B*H <= 1016 at d = 128, B*H <= 2016 at d = 64); larger shapes
 *          return ATTN_ERR_NOMEM and launch nothing.
 *   Set-up: the first call on each device looks up the array's device address
 *          (cudaGetSymbolAddress, with that device current).  Make that first
 *          call before any stream capture.
 *   Sharing: every call on a device uses the same array, which keeps the last
 *          call's contents (no part of it needs to start at zero).  Calls that
 *          overlap on the GPU -- on different streams, or from different host
 *          threads -- race on it and must be serialised by the caller.
 * Other arguments, validation and errors are those of attn_decode, checked in
 * this order: attn_decode's argument checks (ATTN_ERR_NULL, _SHAPE, _HEADDIM,
 * _ARG, _ALIGN, with no CUDA call), then the size limit (ATTN_ERR_NOMEM), then
 * the one-time set-up (ATTN_ERR_CUDA if the address lookup fails).
 */
attn_status attn_decode_noalloc(const void *q, const void *Kcache, const void *Vcache, void *O,
                                int B, int H, int L, int d, float scale, cudaStream_t stream);

/*
 * attn_get_device_status — synchronises `stream`, then reads and clears the
 * library's device status word on the current device.  Returns ATTN_OK, or
 * ATTN_ERR_TIMEOUT if any kernel since the last call gave up on a bounded
 * wait, ATTN_ERR_CUDA if synchronisation itself failed or a kernel could not
 * set up (the forward checks that its dynamic shared memory is 1024-byte
 * aligned and otherwise returns without computing), or ATTN_ERR_ARG if a
 * kernel met an invalid index (a page id).
 */
attn_status attn_get_device_status(cudaStream_t stream);

/* Static, NUL-terminated description of a status code. */
const char *attn_status_string(attn_status status);

/* Most KV splits a decode call uses per head (32): the workspace holds this
 * many partials per head.  Each call picks its own count from the shape (one
 * resident wave of split CTAs for the tensor-core grouped kernel; a power of
 * two from 4 to 32 for the CUDA-core kernels). */
int attn_decode_num_splits(void);

#ifdef __cplusplus
}
#endif

#endif /* EXACT_ATTN_H */
