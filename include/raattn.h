/*
 * libraattn -- rational-softmax (Ra-family) attention for NVIDIA GB300 (sm_103a).
 *
 * C ABI.  Plain pointers and sizes only.  Every device pointer is memory the
 * caller owns (for example from torch, cudaMalloc or a pool); the library keeps
 * no allocation of its own across calls and never frees caller memory.
 *
 * Source of the method: page "Ra-Family: Rational Neural Architecture"
 * (LuminaV-Optimizer docs/nn/README.md), section 3 "Rational Attention &
 * Softmax":
 *   ra_softmax of a row x:  Delta_i = x_max - x_i,  u_i = Delta_i / 16,
 *   q_i = (1 - u_i) / (1 + u_i),  phi_i = q_i^8 for u_i < 1 and exactly 0
 *   otherwise,  p_i = phi_i / sum_j phi_j  (sum_j phi_j >= 1 because the
 *   maximum has phi = 1);  closed-form backward d phi/du = -16 phi / (1 - u^2).
 *   ra_attention:  O = ra_softmax(scale * Q K^T [causal]) V, a drop-in for
 *   scaled_dot_product_attention, computed tile by tile without storing the
 *   [B, H, N_Q, N_K] matrix.
 *
 * Conventions shared by every entry point:
 *   - stream: a cudaStream_t passed as void*; NULL means the legacy default
 *     stream.  Work is enqueued on it and the call returns without waiting.
 *   - Validation happens on the host before anything is launched.  A call
 *     that returns an error status has launched nothing and written nothing.
 *   - Device-side faults are not possible by design; the one device-side
 *     failure is a bounded wait that gave up (RA_ERR_TIMEOUT), which the
 *     kernels record in a library-owned status word and which
 *     ra_device_status() reports.
 *   - No entry point prints, throws or exits.
 *   - Tensors are dense, row-major, contiguous, with every base pointer
 *     16-byte aligned.
 */
#ifndef RAATTN_H
#define RAATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  RA_F32 = 0,   /* IEEE binary32 */
  RA_BF16 = 1   /* bfloat16 */
} ra_dtype_t;

typedef enum {
  RA_OK = 0,
  RA_ERR_ARG = 1,          /* null pointer, size < 1, overflow, misalignment, bad enum */
  RA_ERR_UNSUPPORTED = 2,  /* valid request outside what the library implements */
  RA_ERR_LAUNCH = 3,       /* the CUDA runtime refused the launch or the set-up */
  RA_ERR_TIMEOUT = 4       /* a device-side wait exceeded its limit (see ra_device_status) */
} ra_status_t;

/* Human-readable name of a status code (static string, never NULL). */
const char* ra_status_string(ra_status_t status);

/*
 * ra_softmax_fwd -- y = ra_softmax(x) along the last dimension.
 * Page "Ra-Family: Rational Neural Architecture", section 3, ra_softmax
 * (shift, rational numerator, exact zero for Delta >= 16, normalisation).
 *   x, y     device pointers to rows*cols elements of `dtype`, row-major.  y may
 *            equal x (in place); partial overlap is an error the call cannot see.
 *   rows     >= 1; cols >= 1 (cols == 1 gives p = 1).
 *   dtype    RA_F32, or RA_BF16 (bf16 in and out, fp32 arithmetic, each probability
 *            rounded once to bf16).
 * Errors: RA_ERR_ARG for null pointers, rows/cols < 1, rows*cols overflowing
 * int64, an unknown dtype; RA_ERR_LAUNCH on launch failure.
 */
ra_status_t ra_softmax_fwd(const void* x, void* y, int64_t rows, int64_t cols,
                           ra_dtype_t dtype, void* stream);

/*
 * ra_softmax_bwd -- dx = d/dx sum(dy * ra_softmax(x)) along the last dimension.
 * Page "Ra-Family: Rational Neural Architecture", section 3, ra_softmax,
 * "Closed-Form Backward Pass": from the saved probabilities p = ra_softmax(x)
 * and the shift u = (x_max - x)/16 (recomputed from x), with
 * d phi/du = -16 phi/(1-u^2) and the chain rule through x_max:
 *   dx_j = p_j (dy_j - sum_k p_k dy_k) / (1 - u_j^2)   for j != argmax, u_j < 1
 *   dx_j = 0                                           for u_j >= 1
 *   dx_argmax = -(sum of the other dx_j)               (lowest index among ties)
 *   x, p, dy, dx   device pointers to rows*cols elements of `dtype`; dx may equal dy.
 *   dtype          RA_F32, or RA_BF16: all four arrays bf16, widened exactly to fp32, the
 *                  arithmetic in fp32 and dx rounded once to bf16 (dx_argmax is minus the
 *                  fp32 sum of the others, then rounded).
 * Errors as ra_softmax_fwd.
 */
ra_status_t ra_softmax_bwd(const void* x, const void* p, const void* dy, void* dx,
                           int64_t rows, int64_t cols, ra_dtype_t dtype, void* stream);

/*
 * ra_attention_fwd -- O = ra_softmax(scale * Q K^T [causal]) V, two passes per query tile.
 * Page "Ra-Family: Rational Neural Architecture", section 3, ra_attention
 * (functional form, drop-in for scaled_dot_product_attention; two-pass tiled
 * kernel that skips the V tile whenever every entry of a tile has u >= 1).
 *   q            [B, H, N_Q, D] of in_dtype.
 *   k, v         [B, H, N_K, D] of in_dtype.
 *   o            [B, H, N_Q, D] of out_dtype (written).
 *   row_m        [B, H, N_Q] float: max over allowed keys of the scaled score (written).
 *   row_s        [B, H, N_Q] float: sum of phi over the row, >= 1 (written).
 *   row_arg      [B, H, N_Q] int32: lowest key index attaining the max (written).
 *                row_m, row_s and row_arg are what ra_attention_bwd needs; each may
 *                be NULL when no backward follows.
 *   tile_counts  optional (NULL allowed) int64[2] in device memory, zeroed then written:
 *                [0] = (query tile, key tile) pairs in range (for causal calls, the key
 *                      tiles up to the query tile's diagonal),
 *                [1] = pairs whose P*V product did not run: every entry of the pair lies
 *                      outside the compact support (the V tile is still loaded: the
 *                      decision is taken while it is in flight), or, in masked calls, the
 *                      mask allows no pair of the tile (such tiles are not loaded, and
 *                      take no part in either pass).
 *                Tiles are 128 x 128 on the tensor-core path; at D = 128 with N_Q > 256
 *                two query tiles share each product (CTA pairs), which is skipped
 *                only when both are.
 *   workspace    device memory of ra_attention_fwd_workspace_size() bytes, 16-byte
 *                aligned, contents on entry irrelevant; required for RA_BF16 inputs
 *                (NULL allowed for RA_F32).  The call writes an fp16 copy of v there
 *                (masked calls also two maps of the 128 x 128 tiles: those the mask allows
 *                a pair in, and those it allows every pair of; and per query tile whether
 *                its rows may see exactly a run of leading keys)
 *                and forms P V in fp16, with P rounded to 2^-11 instead of 2^-8.  The
 *                copy is exact for 2^-14 <= |v| <= 65504 (normal fp16); smaller
 *                magnitudes become fp16 subnormals, rounded to a multiple of 2^-24
 *                (below 2^-25 to 0), an absolute error of at most 2^-25 per value.
 *                |v| > 65504 (or NaN) saturates and is reported as RA_ERR_UNSUPPORTED
 *                by ra_device_status().
 *   scale        score scale; <= 0 means 1/sqrt(D).
 *   causal       0: every key visible; nonzero: key j visible to query i iff j <= i
 *                (top-left alignment, as scaled_dot_product_attention's is_causal).
 *   in_dtype     RA_BF16: tensor-core path, D in {64, 128}.
 *                RA_F32: CUDA-core fp32 path (no TF32), D in {16, 32, 64, 128}.
 *   out_dtype    RA_F32 or RA_BF16 for o.
 * Errors: RA_ERR_ARG for null q/k/v/o (or a null workspace with RA_BF16), B, H, N_Q,
 * N_K, D < 1, element counts overflowing int32 indexing per head, a pointer not
 * 16-byte aligned or a bad enum; RA_ERR_UNSUPPORTED for D outside the sets above;
 * RA_ERR_LAUNCH on launch or tensor-map set-up failure.
 */
ra_status_t ra_attention_fwd(const void* q, const void* k, const void* v, void* o,
                             float* row_m, float* row_s, int32_t* row_arg,
                             int64_t* tile_counts, void* workspace,
                             int B, int H, int N_Q, int N_K, int D, float scale, int causal,
                             ra_dtype_t in_dtype, ra_dtype_t out_dtype, void* stream);

/*
 * ra_attention_fwd_workspace_size -- bytes of device workspace ra_attention_fwd (and
 * ra_attention_fwd_masked) needs for these sizes: the fp16 copy of v (B*H*N_K*D*2 bytes,
 * padded to 256), then the two tile maps a masked call builds (each B*H*ceil(N_Q/128)
 * rows of ceil(ceil(N_K/128)/32) uint32 words, padded to 256) and one int32 per row of them
 * (padded to 256).  Returns 0 for invalid sizes.
 */
size_t ra_attention_fwd_workspace_size(int B, int H, int N_Q, int N_K, int D);

/*
 * ra_attention_bwd_workspace_size -- bytes of device workspace ra_attention_bwd needs
 * for these sizes (either input dtype): per (batch*head, 128-row query tile) a block
 * of five 128-entry arrays (two constants of the recomputed weights, D_i = dO_i . O_i,
 * the argmax correction R_i and the argmax index), at least two float arrays of
 * B*H*N_Q entries, then fp16 copies of q, dout, k and v, which the tensor-core path
 * multiplies in fp16 (P, E and dS are then rounded to fp16 rather than bf16 before
 * their products).  The copies are exact for 2^-14 <= |x| <= 65504; smaller values are
 * rounded to a multiple of 2^-24 (fp16 subnormals; below 2^-25 to 0), and |x| > 65504
 * or NaN saturates and is reported as RA_ERR_UNSUPPORTED by ra_device_status().  Last,
 * the two tile maps a masked call builds (tiles with an allowed pair, tiles with every pair
 * allowed), each both ways: B*H*ceil(N_Q/128) rows of ceil(ceil(N_K/128)/32) uint32 words
 * and B*H*ceil(N_K/128) rows of ceil(ceil(N_Q/128)/32), then one int32 per row of either
 * layout.  Each piece is padded to 256 bytes.  Returns 0 for invalid sizes.
 */
size_t ra_attention_bwd_workspace_size(int B, int H, int N_Q, int N_K, int D);

/*
 * ra_attention_bwd -- gradients of sum(dout * O) with respect to q, k and v.
 * Page "Ra-Family: Rational Neural Architecture", section 3, ra_softmax
 * "Closed-Form Backward Pass" (d phi/du = -16 phi/(1-u^2), evaluated from p and
 * u without saved powers of q) and ra_attention ("tiled forward and backward",
 * saved state O(B H N_Q D)).  With P = phi / row_s, dP = dout V^T,
 * D_i = sum_d dout_id O_id and, for allowed j != row_arg_i with u_ij < 1,
 * E_ij = P_ij (dP_ij - D_i) / (1 - u_ij^2), R_i = sum_j E_ij:
 *   dS_ij = E_ij,  dS_{i,row_arg_i} = -R_i,  0 elsewhere;
 *   dq = scale dS K,  dk = scale dS^T Q,  dv = P^T dout.
 *   q, k, v, dout      [B,H,N_Q,D], [B,H,N_K,D], [B,H,N_K,D], [B,H,N_Q,D] of in_dtype.
 *   o                  [B,H,N_Q,D] of o_dtype: the output of ra_attention_fwd.
 *   row_m, row_s, row_arg   the statistics ra_attention_fwd wrote for these inputs
 *                      (all three required).
 *   dq, dk, dv         [B,H,N_Q,D], [B,H,N_K,D], [B,H,N_K,D] of grad_dtype (written).
 *   workspace          device memory of at least ra_attention_bwd_workspace_size()
 *                      bytes, 16-byte aligned; contents on entry do not matter.
 *   o_dtype            dtype of o (RA_F32 or RA_BF16); dout has in_dtype.
 *   grad_dtype         RA_F32 or RA_BF16.
 * Supported combinations and errors as ra_attention_fwd.
 */
ra_status_t ra_attention_bwd(const void* q, const void* k, const void* v, const void* o,
                             const void* dout, const float* row_m, const float* row_s,
                             const int32_t* row_arg, void* dq, void* dk, void* dv,
                             void* workspace,
                             int B, int H, int N_Q, int N_K, int D, float scale, int causal,
                             ra_dtype_t in_dtype, ra_dtype_t o_dtype, ra_dtype_t grad_dtype,
                             void* stream);

/*
 * ra_device_status -- synchronise `stream`, then report and clear the device-side
 * status word of the current device, for everything launched since the last call:
 *   RA_OK               nothing to report;
 *   RA_ERR_TIMEOUT      a kernel gave up a bounded wait (its outputs are undefined);
 *   RA_ERR_UNSUPPORTED  a bf16 (tensor-core) call met an operand beyond the fp16 range
 *                       of its internal copies (|x| > 65504 or NaN: v in the forward;
 *                       q, k, v or dout in the backward); its outputs are undefined;
 *   RA_ERR_LAUNCH       the synchronisation failed, or a kernel found its shared
 *                       memory misaligned and returned without doing anything.
 */
ra_status_t ra_device_status(void* stream);
/*
 * The library looks up the device addresses of its own device variables (this status
 * word, and the scratch array of ra_attention_bwd_noalloc) once per device ordinal and
 * keeps them for the life of the process.  They belong to the device's primary context:
 * after cudaDeviceReset() on a device (or any other destruction of its primary context)
 * they are stale, and the library must not be used on that device again in the process.
 */

/*
 * ra_set_wait_limit_ns -- limit, in nanoseconds of %globaltimer, on every
 * device-side wait of later launches (default 2e9).  0 restores the default.
 * A wait that runs out sets RA_ERR_TIMEOUT and makes the kernel wind down
 * cleanly (in-flight copies drained, tensor memory freed); results are then
 * undefined but the context stays usable.
 */
void ra_set_wait_limit_ns(uint64_t limit_ns);

/*
 * ra_debug_force_timeout -- test knob for the failure path (0 = off, the default).
 * When on, every later tensor-core kernel launch first waits on a barrier that nothing
 * arrives on, so it gives up after the wait limit, winds down as described above and
 * reports RA_ERR_TIMEOUT through ra_device_status().  Results of those calls are undefined.
 */
void ra_debug_force_timeout(int on);

/*
 * ra_debug_fwd_pair -- how later bf16 forward calls with D = 128 are laid out:
 * 0 (default) as CTA pairs (clusters of two CTAs whose tensor-core products span both
 * SMs) when N_Q > 256, otherwise one CTA per pair of query tiles; 1 always single CTAs;
 * 2 always pairs.  Results agree to rounding either way; the knob exists to test and
 * time both layouts.
 */
void ra_debug_fwd_pair(int mode);

/*
 * ra_debug_kernel_events -- measurement knob (n = 0 or events = NULL: off, the default).
 * When on, every later bf16 (tensor-core) ra_attention_fwd / ra_attention_bwd call, masked
 * or not, records the caller's CUDA events (cudaEvent_t handles passed as void*) on its
 * stream at its kernel boundaries, so that each kernel can be timed on the launching
 * stream:
 *   forward:  events[0] before the V conversion, [1] before the attention kernel, [2] after;
 *   backward: events[0] before the operand conversion, [1] before the dQ kernel, [2]
 *             before the dK/dV kernel, [3] after it.
 * At most four events are used; a NULL entry or an index >= n is skipped.  The handles must
 * stay valid while the knob is on.  A failed record makes the call return RA_ERR_LAUNCH.
 */
void ra_debug_kernel_events(void* const* events, int n);

/* Size of the device array behind ra_attention_bwd_noalloc (32 MiB). */
#define RA_NOALLOC_SCRATCH_BYTES (32u << 20)

/*
 * Boolean attention masks (scaled_dot_product_attention's attn_mask: nonzero / true = the
 * query may attend to the key), applied together with `causal`.  Page "Ra-Family: Rational
 * Neural Architecture", section 3, ra_attention (a drop-in for scaled_dot_product_attention).
 * The masked calls take the mask bit-packed: bit (c % 32) of word c / 32 of a row is set when
 * column c may be attended; rows of ra_attention_mask_words(columns) uint32 words (bits of
 * columns past the last are ignored; ra_attention_mask_pack leaves them clear).  A mask has
 * MB x MH heads (MB = 1 or B, MH = 1 or H: shared across the batch and/or the heads); head
 * (b, h) uses mask head (MB > 1 ? b : 0) * MH + (MH > 1 ? h : 0).  A query row with no
 * attendable key gives O = 0, row_s = 0, row_arg = -1 and zero gradients.
 * Masks apply to RA_BF16 inputs (the tensor-core path); with RA_F32 inputs the masked calls
 * return RA_ERR_UNSUPPORTED.
 */

/* ra_attention_mask_words -- uint32 words per packed row of `n` columns (whole 128-column
 * tiles: a multiple of 4); 0 for n < 1. */
int ra_attention_mask_words(int n);

/*
 * ra_attention_mask_pack -- bit-packs a mask of G heads, [G, N_Q, N_K] bytes (row-major,
 * nonzero = may attend), into
 *   mask_q   [G, N_Q, ra_attention_mask_words(N_K)] uint32 (rows = queries), and/or
 *   mask_k   [G, N_K, ra_attention_mask_words(N_Q)] uint32 (the transpose: rows = keys).
 * Either output may be NULL (not both); outputs are 16-byte aligned device memory owned by
 * the caller.  The forward needs mask_q, the backward both.  Errors: RA_ERR_ARG for null
 * pointers, sizes < 1 or misaligned outputs; RA_ERR_LAUNCH on launch failure.
 */
ra_status_t ra_attention_mask_pack(const void* mask, int G, int N_Q, int N_K, uint32_t* mask_q, uint32_t* mask_k,
                                   void* stream);

/*
 * ra_attention_fwd_masked -- ra_attention_fwd with a packed mask (mask_q from
 * ra_attention_mask_pack, MB x MH heads).  Arguments, results and errors otherwise as
 * ra_attention_fwd; RA_ERR_ARG also for a null or misaligned mask_q or MB, MH not in
 * {1, B} x {1, H}.
 */
ra_status_t ra_attention_fwd_masked(const void* q, const void* k, const void* v, void* o, float* row_m,
                                    float* row_s, int32_t* row_arg, int64_t* tile_counts, void* workspace, int B,
                                    int H, int N_Q, int N_K, int D, float scale, int causal, ra_dtype_t in_dtype,
                                    ra_dtype_t out_dtype, const uint32_t* mask_q, int MB, int MH, void* stream);

/*
 * ra_attention_bwd_masked -- ra_attention_bwd for a masked forward: the same packed mask in
 * both layouts (mask_q, mask_k from one ra_attention_mask_pack call), MB x MH heads.
 * Arguments, results and errors otherwise as ra_attention_bwd.
 */
ra_status_t ra_attention_bwd_masked(const void* q, const void* k, const void* v, const void* o, const void* dout,
                                    const float* row_m, const float* row_s, const int32_t* row_arg, void* dq,
                                    void* dk, void* dv, void* workspace, int B, int H, int N_Q, int N_K, int D,
                                    float scale, int causal, ra_dtype_t in_dtype, ra_dtype_t o_dtype,
                                    ra_dtype_t grad_dtype, const uint32_t* mask_q, const uint32_t* mask_k, int MB,
                                    int MH, void* stream);

/*
 * ra_attention_bwd_noalloc -- ra_attention_bwd without a caller-supplied workspace.
 * The pages have no counterpart: this entry point exists for callers that cannot
 * allocate device memory, such as code inside a framework that owns the allocator and
 * offers no temporary buffers, or a host path where cudaMalloc (which may synchronise
 * the device) is not allowed.  The workspace comes instead from a fixed array of
 * RA_NOALLOC_SCRATCH_BYTES inside the library: every GPU that loads the library holds
 * that memory until the process exits, and nothing is allocated per call.
 *   Arguments, results and errors are those of ra_attention_bwd without `workspace`.
 *   Sizes whose workspace exceeds RA_NOALLOC_SCRATCH_BYTES are rejected with
 *   RA_ERR_UNSUPPORTED before anything runs (use ra_attention_bwd then).  The workspace
 *   counted is the one this call's path uses: ra_attention_bwd_workspace_size() for
 *   RA_BF16 inputs, and for RA_F32 inputs only two float arrays of B*H*N_Q entries (each
 *   padded to 256 bytes).  Device ordinals of 64 and above also give RA_ERR_UNSUPPORTED.
 *   The first call on a device looks up the array's device address (once per device)
 *   and keeps it, like the status word's (see ra_device_status); make that first call
 *   before any stream capture.
 *   All calls share the one array and it keeps the previous call's contents (nothing in
 *   it needs to start at zero).  Calls that overlap on the GPU -- on different streams,
 *   or from different host threads without ordering -- race on it: serialise them.
 */
ra_status_t ra_attention_bwd_noalloc(const void* q, const void* k, const void* v, const void* o,
                                     const void* dout, const float* row_m, const float* row_s,
                                     const int32_t* row_arg, void* dq, void* dk, void* dv,
                                     int B, int H, int N_Q, int N_K, int D, float scale, int causal,
                                     ra_dtype_t in_dtype, ra_dtype_t o_dtype, ra_dtype_t grad_dtype,
                                     void* stream);

#ifdef __cplusplus
}
#endif

#endif /* RAATTN_H */
