/*
 * fa_back.h -- C ABI of the GB300 (sm_103a) flash-attention backward over a raw K/V cache.
 *
 * The operation is ggml's FLASH_ATTN_BACK as described in "CUDA: FLASH_ATTN_BACK kernels"
 * (CambrianTech/llama.cpp pull request 63; review of the first revision, "The math in
 * fattn_back_q / fattn_back_kv"):
 *
 *   hk       = h / (H / Hkv)                                  GQA map
 *   allowed  = (mask == NULL or mask[h % Hm][i][j] != -inf) and (!causal or j <= M - N + i)
 *   s_ij     = scale * q_i . k^_j + mask[h % Hm][i][j]
 *   lse_ih   = log sum_{allowed j} exp(s_ij)                  (-inf when no key is allowed)
 *   p_ij     = exp(s_ij - lse_ih)                             (0 when not allowed)
 *   delta_ih = sum_j p_ij (dO_i . v^_j)                       (= rowsum(dO o O), O never formed)
 *   dS_ij    = p_ij (dO_i . v^_j - delta_ih)
 *   dQ_i     = scale sum_j dS_ij k^_j
 *   dK_j     = scale sum_{h in group(hk), i} dS_ij q_i
 *   dV_j     = sum_{h in group(hk), i} p_ij dO_i
 *
 * k^ and v^ are decoded from the cache rows exactly as their block formats define (see
 * fa_type).  The N x M score matrix is never materialised.  Fully masked rows give
 * lse = -inf, delta = 0 and a zero dQ row (same review, "Masking and q8_0").
 *
 * Layouts (all row-major, the last index fastest; element sizes in parentheses):
 *   q      [N][H][D]        f32     dO    [N][H][Dv]      f32
 *   k      [M][Hkv][row_k]  raw     v     [M][Hkv][row_v] raw     (row = fa_row_bytes(type, D))
 *   mask   [Hm][N][M]       IEEE binary16 bits; element (key j, query i, head hm) at
 *                           (hm*N + i)*M + j  (ggml's [M, N, Hm] order); Hm = 1 or H
 *   dQ     [N][H][D]        f32     dK    [M][Hkv][D]     f32     dV [M][Hkv][Dv] f32
 *   lse    [N][H]           f32 (natural log)             delta [N][H] f32
 *
 * Ownership: every pointer is caller-owned DEVICE memory on the current device, including the
 * workspace.  The library allocates no device memory and keeps no reference after return.
 *
 * Asynchrony: fa_back() validates its arguments on the host, enqueues its kernels on `stream`
 * and returns without synchronising.  Outputs are valid once the stream's work completes.  A
 * call may be captured into a CUDA graph (stream capture): its host work runs at the call and
 * only kernel launches are enqueued, so a replay reruns the backward on the same buffers.
 *
 * Errors: argument errors are reported before anything is enqueued and leave the outputs
 * untouched.  A launch failure returns FA_ERR_CUDA.  A kernel that gives up on a bounded wait
 * records FA_ERR_TIMEOUT in a device word that fa_back_get_error() reads after the caller has
 * synchronised; before it exits it waits (again bounded) for its own loads and tensor-core
 * products still in flight and frees its tensor memory, so the context stays usable.
 *
 * Determinism: every output element has exactly one writer and every sum runs in a fixed
 * order, so repeated calls with the same inputs give bit-identical outputs.
 */
#ifndef FA_BACK_H
#define FA_BACK_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Cache row formats.
 *   FA_F32  : D IEEE binary32 values.
 *   FA_F16  : D IEEE binary16 values.
 *   FA_Q8_0 : D/32 blocks of 34 bytes: binary16 scale d, then 32 int8 codes; value = code * d.
 *   FA_Q4_0 : D/32 blocks of 18 bytes: binary16 scale d, then 16 bytes; byte b holds element b
 *             in its low nibble and element b+16 in its high nibble; value = (nibble - 8) * d.
 * The q8_0 block follows the review's description of the kernel's q8_0 load (pull request 63);
 * the q4_0 block is the raw-cache format the forward kernel of torad-labs/llama.cpp pull
 * request 71 reads.  Rows of the cache are contiguous blocks. */
typedef enum { FA_F32 = 0, FA_F16 = 1, FA_Q8_0 = 2, FA_Q4_0 = 3 } fa_type;

typedef enum {
  FA_OK = 0,
  FA_ERR_NULL = 1,        /* a required pointer is NULL (mask may be NULL)                     */
  FA_ERR_TYPE = 2,        /* k_type or v_type is not an fa_type                                 */
  FA_ERR_SHAPE = 3,       /* N, M < 0; H, Hkv < 1; H % Hkv != 0; mask_heads not 1 or H         */
  FA_ERR_ALIGN = 4,       /* a pointer is not 16-byte aligned (workspace: 256-byte aligned)     */
  FA_ERR_UNSUPPORTED = 5, /* D or Dv not in {64, 128, 256}; size limits exceeded                */
  FA_ERR_DEVICE = 6,      /* the current device is not compute capability 10.3                  */
  FA_ERR_CUDA = 7,        /* a CUDA runtime call or kernel launch failed                        */
  FA_ERR_TIMEOUT = 8,     /* a kernel gave up on a bounded wait (see fa_back_get_error)         */
  FA_ERR_WORKSPACE = 9    /* workspace is NULL or smaller than fa_back_workspace_size_min()     */
} fa_status;

/* Bytes in one cache row of `type` holding D values (-1 if D does not fit the format). */
long fa_row_bytes(int type, int D);

/* Workspace bytes of fa_back()'s fastest plan on the current device for this shape.  Beside the
 * per-row statistics and split partials, that plan holds binary16 copies of the decoded K and V
 * cache (2 * Hkv * M * (D + Dv) bytes) and the binary16 dS of every row and key (2 * N * H * M'
 * bytes, M' = M rounded up to 64), from which dQ is one product.  A workspace too small for both
 * gets the next fastest plan that fits: the stored dS without the copies (every pass then decodes
 * the raw cache tiles in shared memory), else the copies alone (dS recomputed in a dQ pass). */
size_t fa_back_workspace_size(int N, int M, int H, int Hkv, int D, int Dv);

/* The smallest workspace fa_back() accepts for this shape: its plan decodes the raw cache inside
 * the row passes and does not split the keys.  A workspace between the two sizes gets the
 * fastest plan that fits it; one plan and its results are fixed by the shape and
 * workspace_bytes, so equal calls give bit-identical outputs. */
size_t fa_back_workspace_size_min(int N, int M, int H, int Hkv, int D, int Dv);

/* The plan fa_back() runs for this shape and workspace_bytes on the current device (an SM count
 * of 152 when no device is visible): *level 2 (binary16 K'/V' copies and the stored dS), 3 (the
 * stored dS, raw rows decoded in the passes), 1 (the copies only) or 0 (raw rows decoded in the
 * passes, dS recomputed in a dQ pass), the number of key splits of its row
 * passes, and the workspace bytes it uses.  Host only: nothing is enqueued.  FA_ERR_WORKSPACE
 * when workspace_bytes is below fa_back_workspace_size_min(); FA_ERR_SHAPE / FA_ERR_UNSUPPORTED
 * as for fa_back().  Any output pointer may be NULL. */
fa_status fa_back_plan_info(int N, int M, int H, int Hkv, int D, int Dv, size_t workspace_bytes, int* level,
                            int* key_splits, size_t* plan_bytes);

/*
 * The backward.  scale multiplies q.k before the mask is added (the reading used for the
 * pages' tests is scale = 1/sqrt(D)).  causal != 0 applies the causal tail j <= M - N + i.
 * mask may be NULL; mask_heads (Hm) is ignored then.  Every element of dQ, dK, dV, lse and
 * delta is written.  Pointers: q, dO, dQ, dK, dV, lse, delta and mask 16-byte aligned; k, v
 * 16-byte aligned; workspace 256-byte aligned.
 */
fa_status fa_back(const float* q, const void* k, int k_type, const void* v, int v_type,
                  const uint16_t* mask, int mask_heads, const float* dO, float scale, int N, int M,
                  int H, int Hkv, int D, int Dv, int causal, float* dQ, float* dK, float* dV,
                  float* lse, float* delta, void* workspace, size_t workspace_bytes, void* stream);

/*
 * fa_back() for a caller that already has the row statistics of the forward pass: lse [N][H]
 * (natural log, -inf for a row with no allowed key) and delta [N][H] = rowsum(dO o O) with O the
 * forward output.  The backward then skips its LSE/D pass (the QK^T and dO V^T products over every
 * pair that only serve those statistics) and writes dQ, dK and dV only; every other argument is
 * as for fa_back().  lse and delta are read, 16-byte aligned, and must come from the same
 * Q, K, V, mask, scale and causal setting (the gradients are exact for the statistics given).
 * With N > 0, NULL lse or delta is FA_ERR_NULL.
 */
fa_status fa_back_with_stats(const float* q, const void* k, int k_type, const void* v, int v_type,
                             const uint16_t* mask, int mask_heads, const float* dO, const float* lse,
                             const float* delta, float scale, int N, int M, int H, int Hkv, int D, int Dv,
                             int causal, float* dQ, float* dK, float* dV, void* workspace,
                             size_t workspace_bytes, void* stream);

/*
 * fa_back() restricted to the plans that keep no decoded copy of the cache: every K and V tile is
 * read as raw cache rows and decoded in shared memory by the pass that uses it.  With a workspace
 * of at least fa_back_workspace_size_nocopy() bytes the plan stores dS (level 3: dQ is one product
 * over it, decoding raw K tiles once per two row tiles); with less, down to
 * fa_back_workspace_size_min(), it recomputes dS in a dQ pass (level 0).  Arguments, results,
 * errors and determinism as for fa_back().
 */
size_t fa_back_workspace_size_nocopy(int N, int M, int H, int Hkv, int D, int Dv);
fa_status fa_back_nocopy(const float* q, const void* k, int k_type, const void* v, int v_type,
                         const uint16_t* mask, int mask_heads, const float* dO, float scale, int N, int M,
                         int H, int Hkv, int D, int Dv, int causal, float* dQ, float* dK, float* dV,
                         float* lse, float* delta, void* workspace, size_t workspace_bytes, void* stream);

/*
 * fa_back() with three score extensions that the operation above does not have.  The pull request
 * this library follows lists ALiBi, soft-capping and sink gradients among the features it does
 * not support and defines none of them; the definitions taken here are the usual ones:
 *   x_ij   = scale * q_i . k^_j
 *   s_ij   = c tanh(x_ij / c)    (softcap = c > 0: the logit soft-capping of the Gemma 2 models)
 *            or x_ij             (softcap = 0)
 *            + mask[h % Hm][i][j]
 *            + alibi_slopes[h] * (j - (M - N + i))   (ALiBi, Press, Smith and Lewis, "Train Short,
 *              Test Long": 0 on the causal diagonal, falling linearly with the distance to
 *              earlier keys; M - N + i is query i's position on the key axis, as for causal)
 *   lse_ih = log(exp(sinks[h]) + sum_{allowed j} exp(s_ij))   (a sink: one logit per head that
 *            joins every row's softmax denominator and has no value row)
 *   p_ij, delta_ih as in fa_back() with this lse (the keys' weights sum to 1 - exp(sinks[h] - lse))
 *   dS_ij  = p_ij (dO_i . v^_j - delta_ih) (1 - tanh^2(x_ij / c))   (the last factor 1 without a cap)
 *   dQ, dK, dV as in fa_back() with this dS;  dsinks[h] = -sum_i exp(sinks[h] - lse_ih) delta_ih.
 * alibi_slopes [H] and sinks [H] are f32 device arrays, or NULL for none; softcap must be >= 0
 * and finite (else FA_ERR_SHAPE).  dsinks [H] (f32, device) is written when sinks is given and
 * may then be NULL (no sink gradient); it is ignored without sinks.  These pointers need 4-byte
 * alignment.  With sinks, a row without an allowed key has lse = sinks[h], delta = 0 and a zero
 * dQ row.  All four NULL / 0 is fa_back() itself: the same plan and bit-identical results.
 * Workspace, plan, asynchrony and the other errors are those of fa_back().
 */
fa_status fa_back_ext(const float* q, const void* k, int k_type, const void* v, int v_type,
                      const uint16_t* mask, int mask_heads, const float* dO, float scale, int N, int M, int H,
                      int Hkv, int D, int Dv, int causal, const float* alibi_slopes, float softcap,
                      const float* sinks, float* dsinks, float* dQ, float* dK, float* dV, float* lse,
                      float* delta, void* workspace, size_t workspace_bytes, void* stream);

/*
 * The forward of the same attention over the raw cache: O [N][H][Dv] = softmax(scale * q k^T +
 * mask, causal tail) v and lse [N][H] (natural log), f32.  A row without an allowed key gets
 * O = 0 and lse = -inf.  Arguments as for fa_back(); O and lse are written, 16-byte aligned.
 * The lse it writes, with delta = rowsum(dO o O), is what fa_back_with_stats() takes.
 * Computation: one pass per row tile with an online softmax (O accumulated against a running
 * maximum and rescaled when that maximum moves; binary16 operands as in the backward), key
 * splits merged in a fixed order.  The result does not depend on timing.
 */
size_t fa_forward_workspace_size(int N, int M, int H, int Hkv, int D, int Dv);
fa_status fa_forward(const float* q, const void* k, int k_type, const void* v, int v_type,
                     const uint16_t* mask, int mask_heads, float scale, int N, int M, int H, int Hkv,
                     int D, int Dv, int causal, float* O, float* lse, void* workspace,
                     size_t workspace_bytes, void* stream);

/*
 * B independent backwards of the same shape (a leading batch dimension, ggml's ne[3]): q, dO,
 * dQ [B][N][H][·]; k, v, dK, dV [B][M][Hkv][·]; lse, delta [B][N][H]; the mask [B][Hm][N][M]
 * when mask_per_batch != 0, else one [Hm][N][M] shared by every batch.  All tensors contiguous.
 * Batch b runs as fa_back() on its slices, one after another on `stream`, sharing the workspace
 * (fa_back_workspace_size() of one problem suffices); every slice must meet fa_back()'s
 * alignment.  The first failing batch's status is returned (earlier batches are enqueued).
 */
fa_status fa_back_batched(int B, const float* q, const void* k, int k_type, const void* v, int v_type,
                          const uint16_t* mask, int mask_heads, int mask_per_batch, const float* dO,
                          float scale, int N, int M, int H, int Hkv, int D, int Dv, int causal, float* dQ,
                          float* dK, float* dV, float* lse, float* delta, void* workspace,
                          size_t workspace_bytes, void* stream);

/*
 * Input strides for fa_back_strided().  The operator keeps its outer strides and its q / dO
 * component strides ("CUDA: FLASH_ATTN_BACK kernels", CambrianTech/llama.cpp pull request 63,
 * PR description), so each input may be a view:
 *   Q  element (i, h, c) at q[i*q_row + h*q_head + c*q_comp]       (f32 elements)
 *   dO element (i, h, c) at dO[i*do_row + h*do_head + c*do_comp]   (f32 elements)
 *   K  row (j, hk) starts at (const char*)k + j*k_cell + hk*k_head  (bytes; a row's fa_row_bytes
 *      bytes are contiguous, since a block is the format's unit; v likewise with v_cell, v_head)
 *   mask element (j, i, hm) at word hm*mask_head + i*mask_row + j    (FA_MASK_F16: binary16 words)
 *      or bit j % 32 of word hm*mask_head + i*mask_row + j / 32      (FA_MASK_BITS: 32-bit words)
 * Every stride is >= 0 (0 repeats one element, a broadcast view); the K and V byte strides are
 * even.  The contiguous layouts of fa_back() are q_row = H*D, q_head = D, q_comp = 1,
 * k_cell = Hkv*fa_row_bytes(k_type, D), k_head = fa_row_bytes(k_type, D), mask_head = N*M (F16)
 * and mask_row = M.
 */
typedef struct fa_strides {
  int64_t q_row, q_head, q_comp;
  int64_t do_row, do_head, do_comp;
  int64_t k_cell, k_head;
  int64_t v_cell, v_head;
  int64_t mask_head, mask_row;
} fa_strides;

/* Mask formats of fa_back_strided().  FA_MASK_F16: binary16 additive values, as for fa_back().
 * FA_MASK_BITS: one bit per (query, key), set = the key is allowed (adds +0), clear = masked
 * (-inf); the mask the raw-cache forward of torad-labs/llama.cpp pull request 71 reads is
 * bit-packed, and this is the plainest reading of one, since that page gives no bit order. */
#define FA_MASK_F16 0
#define FA_MASK_BITS 1

/* Workspace bytes of fa_back_strided() with fa_back()'s fastest plan: contiguous copies of Q, dO,
 * K, V and (mask_heads > 0) a binary16 mask, each rounded up to 256 bytes, followed by
 * fa_back_workspace_size().  0 for invalid arguments. */
size_t fa_back_strided_workspace_size(int N, int M, int H, int Hkv, int D, int Dv, int k_type, int v_type,
                                      int mask_heads);

/*
 * fa_back() on inputs given as views (strides in *strides) and with a binary16 or bit-packed
 * mask (mask_format).  Each input is copied once, on `stream`, into a contiguous region at the
 * front of the workspace (the mask's bits widened to binary16 0 / -inf), then fa_back() runs on
 * those regions with the rest of the workspace, so its plan, results and determinism are those
 * of fa_back() given workspace_bytes minus the copies.  The outputs are contiguous, laid out as
 * for fa_back().  Pointers: q, dO 4-byte aligned; k, v 2-byte aligned; the mask 2-byte
 * (FA_MASK_F16) or 4-byte (FA_MASK_BITS) aligned; outputs 16-byte aligned; workspace 256-byte
 * aligned.  Errors as for fa_back(), plus: strides NULL is FA_ERR_NULL; a negative stride or an
 * unknown mask_format is FA_ERR_SHAPE; an odd K/V byte stride is FA_ERR_ALIGN; a workspace
 * smaller than the copies plus fa_back_workspace_size_min() is FA_ERR_WORKSPACE.  Every element a
 * view addresses must lie inside memory the caller owns; the library cannot check that.
 */
fa_status fa_back_strided(const float* q, const void* k, int k_type, const void* v, int v_type,
                          const void* mask, int mask_format, int mask_heads, const float* dO,
                          const fa_strides* strides, float scale, int N, int M, int H, int Hkv, int D,
                          int Dv, int causal, float* dQ, float* dK, float* dV, float* lse, float* delta,
                          void* workspace, size_t workspace_bytes, void* stream);

/* Sticky device-side status of the kernels enqueued so far on the current device
 * (FA_OK or FA_ERR_TIMEOUT).  Synchronises the device, then clears the word. */
fa_status fa_back_get_error(void);

/* Human-readable name of a status code. */
const char* fa_back_status_string(int status);

/*
 * Measurement hook (not part of the operation).  fa_back_profile(1) makes the following
 * fa_back() calls on this process record a CUDA event after each of their kernel launches
 * (at most 256 calls are recorded; later calls run unrecorded).  fa_back_profile(0) stops.
 * fa_back_profile_read() synchronises on the recorded events and writes, for each kernel of
 * the launch sequence, the summed device time in ms (ms_sum[k]) and the number of recorded
 * launches (launches[k]); names[k] receives a static string naming the kernel.  It returns the
 * number of kernels written (at most max_kernels) and clears the record.  The events are
 * created on first use and kept until process exit; no device memory is allocated.
 */
fa_status fa_back_profile(int enable);
int fa_back_profile_read(float* ms_sum, int* launches, const char** names, int max_kernels);

/*
 * fa_back() for callers that cannot allocate device memory.  "CUDA: FLASH_ATTN_BACK kernels"
 * defines no such entry point: its operator takes no workspace argument at all.  Some callers cannot hand the library a
 * workspace: graph executors that own every device buffer through their own pool and give an
 * operator no scratch pointer, and services that allocate nothing once they are set up.  This
 * entry point takes the same arguments as fa_back() minus the workspace and uses instead one
 * file-scope device array of FA_NOALLOC_SCRATCH_BYTES (64 MiB), which every GPU that loads the
 * library holds until the process exits.  It calls no cudaMalloc, cudaFree or other allocating
 * routine; the caller still passes every input and output.
 *   - The plan is fa_back()'s for a workspace of FA_NOALLOC_SCRATCH_BYTES: the fastest that
 *     fits.  Problems whose fa_back_workspace_size_min() exceeds it are rejected with
 *     FA_ERR_WORKSPACE before anything is enqueued.
 *   - Every call looks up the array's device address in the current device's context (the
 *     module, and the array with it, is loaded in each context that first uses the library).
 *   - Every call on a device shares the one array, which keeps the last call's contents.
 *     Nothing in it needs to start at zero: each call writes every scratch word before reading
 *     it.  Calls whose work overlaps on the GPU (other streams, other threads) race on the
 *     array; serialise them.
 */
#define FA_NOALLOC_SCRATCH_BYTES (64ull << 20)
fa_status fa_back_noalloc(const float* q, const void* k, int k_type, const void* v, int v_type,
                          const uint16_t* mask, int mask_heads, const float* dO, float scale, int N,
                          int M, int H, int Hkv, int D, int Dv, int causal, float* dQ, float* dK,
                          float* dV, float* lse, float* delta, void* stream);

/*
 * Exercises the failure-detection path of the bounded waits without a fault: enqueues one
 * kernel on `stream` whose thread waits up to `limit_ns` nanoseconds (0 < limit_ns <= 2 s) on
 * an mbarrier that nothing completes, records FA_ERR_TIMEOUT in the device error word exactly as
 * the backward's kernels do when a wait runs out, and returns.  The context stays usable;
 * fa_back_get_error() then reports FA_ERR_TIMEOUT once (and clears it).  Returns FA_OK when
 * the kernel was enqueued, FA_ERR_SHAPE for a limit outside that range.
 */
fa_status fa_back_selftest_timeout(unsigned long long limit_ns, void* stream);

/*
 * Failure-detection hook for the real passes (not part of the operation).  The kernels of the
 * next call that validates its arguments and runs the passes (fa_back(), fa_back_ext(),
 * fa_back_with_stats(), fa_forward(), or an entry point built on them) give up on every wait
 * that lasts longer than limit_ns nanoseconds (0: on every wait not complete at once) instead of
 * after 2 s.  They then take the path of a real stall: FA_ERR_TIMEOUT is recorded in the device
 * error word, each CTA stops issuing work, waits (up to 2 s) for its own loads and tensor-core
 * products still in flight, frees its tensor memory and exits.  That call's outputs are
 * undefined; later calls use the normal limit.  Returns FA_OK, or FA_ERR_SHAPE for a limit
 * above 2 s.
 */
fa_status fa_back_test_wait_limit(unsigned long long limit_ns);

#ifdef __cplusplus
}
#endif

#endif /* FA_BACK_H */
