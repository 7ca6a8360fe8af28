/*
 * libattn -- multi-head scaled-dot-product attention for NVIDIA GB300 (sm_103a).
 *
 * The operation, in every entry point, for each query row i and its admitted
 * key set K(i):
 *     S = Q K^T * scale,  P = row softmax(S) over K(i),  O = P V
 * ("cuBLAS matmuls for ... attention scores" plus a softmax kernel, iris.c
 * issue #15 "CUDA codepath !"; the windowed score / softmax / accumulate of
 * candle PR #11's neighborhood attention; the single-token decode attention
 * over a device-resident KV cache of fak "GPU - the in-kernel forward pass",
 * sections 0 and 4).
 *
 * Conventions shared by all entry points
 *   - Tensors are DEVICE pointers to contiguous row-major arrays with the head
 *     dimension innermost.  Attention tensors are heads-major [B, H, N, D].
 *   - dtype ATTN_F32: float32 storage, exact fp32 FMA arithmetic (no TF32).
 *     dtype ATTN_BF16 / ATTN_F16: bfloat16 / IEEE half storage (candle's
 *     F32 / BF16 / F16 trio); the contractions run on the tensor cores
 *     (tcgen05) with fp32 accumulation where the shapes allow (else the exact
 *     SIMT kernel), the softmax in fp32, P rounded to the storage type for the
 *     P V product; the output is rounded to the storage type (to nearest even).
 *   - D (head dimension) is 32, 64 or 128.
 *   - scale <= 0 selects 1/sqrt(D).
 *   - Inputs are never written.  The output must not alias any input.
 *   - The caller owns every buffer.  No entry point allocates device memory
 *     and none synchronises: work is enqueued on `stream` (a cudaStream_t;
 *     NULL = the legacy default stream) and the call returns.
 *   - Errors: arguments are validated on the host before any launch; a failed
 *     check returns ATTN_ERR_INVALID_ARG / ATTN_ERR_UNSUPPORTED /
 *     ATTN_ERR_RESOURCE and launches nothing.  A launch failure returns
 *     ATTN_ERR_CUDA.  Device-side waits are bounded: a wait that runs out sets
 *     a device error word that attn_device_status() reports.  Nothing is
 *     thrown across this interface.
 *   - Thread safety: calls may come from several host threads; each call only
 *     reads its arguments and enqueues work.
 */
#ifndef LIBATTN_H
#define LIBATTN_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define ATTN_API __attribute__((visibility("default")))
#else
#define ATTN_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    ATTN_F32 = 0,
    ATTN_BF16 = 1,
    ATTN_F16 = 2
} attn_dtype_t;

typedef enum {
    ATTN_OK = 0,
    ATTN_ERR_INVALID_ARG = 1,   /* null pointer, bad shape, bad kernel, ...       */
    ATTN_ERR_UNSUPPORTED = 2,   /* valid request this build has no kernel for     */
    ATTN_ERR_RESOURCE = 3,      /* shared memory / workspace too small            */
    ATTN_ERR_CUDA = 4,          /* a CUDA runtime call or launch failed           */
    ATTN_ERR_TIMEOUT = 5,       /* a bounded device wait ran out (device word)    */
    ATTN_ERR_DEVICE_CHECK = 6   /* a device-side consistency check failed         */
} attn_status_t;

/*
 * Full (unmasked, non-causal) attention.
 *   q [B, H, Nq, D], k and v [B, H, Nkv, D], o [B, H, Nq, D]; dtype for all.
 *   Every query attends to all Nkv keys of its (batch, head).
 *   Requires B, H, Nq, Nkv >= 1 and D in {32, 64, 128}.
 * Passage: iris.c issue #15, the reply listing "attention scores" among the
 * cuBLAS matmuls and softmax among the custom kernels.
 */
ATTN_API attn_status_t attn_full_fwd(const void *q, const void *k, const void *v, void *o,
                            int B, int H, int Nq, int Nkv, int D,
                            attn_dtype_t dtype, float scale, void *stream);

/*
 * Full attention on strided views: the operation of attn_full_fwd, with each
 * of q, k, v and o addressed through its own element strides instead of the
 * contiguous [B, H, N, D] layout, so that transposed [B, N, H, D] tensors,
 * slices of a packed QKV projection or a column block of a wider output are
 * used in place, with no copy.
 *   x_strides[3] = element strides of (batch, head, row); D is contiguous
 *   (stride 1).  Element (b, h, n, d) of x is x[b*s[0] + h*s[1] + n*s[2] + d].
 *   Every stride is >= 1 and a multiple of 16 bytes (8 elements for bf16 and
 *   f16, 4 for f32), as the tensor-memory-access unit requires; a stride
 *   whose extent is 1 is ignored.  Base pointers are 16-byte aligned.
 *   q, k and v are read only and may overlap one another; o must not
 *   overlap them, and its (batch, head, row) rows must be disjoint (checked:
 *   sorted by stride, each stride covers the extent below it).
 *   Same sizes, dtypes, scale and status codes as attn_full_fwd.
 * Passage: the unmasked attention of attn_full_fwd; the layout is an
 * addressing choice with no counterpart in the pages.
 */
ATTN_API attn_status_t attn_full_fwd_strided(const void *q, const void *k, const void *v,
                                            void *o, int B, int H, int Nq, int Nkv, int D,
                                            const int64_t q_strides[3],
                                            const int64_t k_strides[3],
                                            const int64_t v_strides[3],
                                            const int64_t o_strides[3],
                                            attn_dtype_t dtype, float scale, void *stream);

/*
 * Joint text+image attention with a multi-axis rotary embedding on Q and K.
 *   q, k, v, o [B, H, N, D]; N = text + image tokens in the caller's order.
 *   pos: DEVICE int32 [N, 4], the 4 position ids of each token.
 *   axes_dim: HOST int[4], channel widths of the 4 axis blocks; each even and
 *   sum == D.  In the block of axis a starting at channel c_a, the adjacent
 *   pair (c_a + 2i, c_a + 2i + 1) rotates by phi = pos[t][a] * theta^(-2i/axes_dim[a]):
 *       x0' = x0 cos(phi) - x1 sin(phi),   x1' = x0 sin(phi) + x1 cos(phi).
 *   V is not rotated.  Then full attention over all N tokens.
 *   workspace: DEVICE scratch of at least attn_rope_joint_workspace_bytes(...)
 *   bytes, 256-byte aligned, that no other call uses concurrently; the rotated
 *   copies of Q and K (in the storage dtype) live there during the call.
 * Passage: iris.c issue #15, GGML lessons item 3 (FLUX's custom RoPE: 4 axes
 * [32,32,32,32], separate text/image positions, repeat_interleave) and the
 * closing "AdaLN + custom RoPE + joint attention" remark.
 */
ATTN_API attn_status_t attn_rope_joint_fwd(const void *q, const void *k, const void *v, void *o,
                                  int B, int H, int N, int D,
                                  const int32_t *pos, const int axes_dim[4], float theta,
                                  attn_dtype_t dtype, float scale,
                                  void *workspace, size_t workspace_bytes, void *stream);

ATTN_API size_t attn_rope_joint_workspace_bytes(int B, int H, int N, int D, attn_dtype_t dtype);

/*
 * Causal grouped-query prefill (self-attention over a prompt).
 *   q, o [B, Hq, N, D]; k, v [B, Hkv, N, D]; Hq % Hkv == 0.  Query head hq
 *   reads KV head hq / (Hq / Hkv); query position i attends to key positions
 *   j <= i.  bf16 and f16 run on the tensor cores for D in {64, 128}; fp32
 *   (and the 16-bit types with D = 32) on the exact-FFMA SIMT kernel.
 * Passage: fak "GPU - the in-kernel forward pass", section 3 (Llama prefill
 * workloads pp64 .. pp512 of a grouped-query model).
 */
ATTN_API attn_status_t attn_causal_gqa_fwd(const void *q, const void *k, const void *v, void *o,
                                           int B, int Hq, int Hkv, int N, int D,
                                           attn_dtype_t dtype, float scale, void *stream);

/*
 * Causal grouped-query prefill on strided views: the operation of
 * attn_causal_gqa_fwd with q, k, v and o addressed through element strides
 * of (batch, head, row) as in attn_full_fwd_strided (D contiguous, every
 * stride a multiple of 16 bytes, extent-1 axes' strides ignored, o's rows
 * disjoint), so a Llama layer's [B, N, Hq, D] query projection and a packed
 * [B, N, 2, Hkv, D] key/value projection are read in place.
 * Passage: as attn_causal_gqa_fwd; the layout is an addressing choice with
 * no counterpart in the pages.
 */
ATTN_API attn_status_t attn_causal_gqa_fwd_strided(const void *q, const void *k, const void *v,
                                                  void *o, int B, int Hq, int Hkv, int N, int D,
                                                  const int64_t q_strides[3],
                                                  const int64_t k_strides[3],
                                                  const int64_t v_strides[3],
                                                  const int64_t o_strides[3],
                                                  attn_dtype_t dtype, float scale, void *stream);

/*
 * Single-token grouped-query decode attention over a KV cache.
 *   q [B, Hq, D], o [B, Hq, D]; k_cache, v_cache [B, Hkv, Lmax, D].
 *   seq_len: DEVICE int32 [B], 1 <= seq_len[b] <= Lmax (checked on the device;
 *   a violation sets ATTN_ERR_DEVICE_CHECK and that batch's output is left
 *   unwritten).  Query head hq reads KV head hq / (Hq / Hkv) and attends to
 *   cache rows j < seq_len[b]; rows at or beyond seq_len[b] are never used.
 *   Requires Hq % Hkv == 0, Hq / Hkv in {1, 2, 4, 8}, D in {64, 128}, dtype
 *   ATTN_BF16 or ATTN_F16 (q, caches and o alike).
 *   workspace: DEVICE scratch of attn_decode_gqa_workspace_bytes(...) bytes,
 *   256-byte aligned, ZERO-FILLED before its first use.  It holds per-split
 *   partial results and per-(batch, kv-head) arrival counters when the splits
 *   merge through global memory; when the splits of every (batch, kv-head)
 *   fit on the GPU at once as thread-block clusters they merge through
 *   distributed shared memory instead and the workspace is not touched.
 *   Every call that completes leaves the counters at zero, so the same workspace serves
 *   the next call without clearing.  Calls that share a workspace must not
 *   overlap on the GPU.  After a call that reported a device error, zero it
 *   again.
 * Passage: fak "GPU - the in-kernel forward pass", section 0 (device-resident
 * KV cache) and section 4 (naive decode attention: per-call scratch, one block
 * per head, no flash/paged attention).
 */
ATTN_API attn_status_t attn_decode_gqa(const void *q, const void *k_cache, const void *v_cache,
                              const int32_t *seq_len, void *o,
                              int B, int Hq, int Hkv, int Lmax, int D,
                              attn_dtype_t dtype, float scale,
                              void *workspace, size_t workspace_bytes, void *stream);

ATTN_API size_t attn_decode_gqa_workspace_bytes(int B, int Hq, int Hkv, int Lmax, int D);

/*
 * attn_decode_gqa without a workspace argument, for callers that cannot hand
 * this library any device memory beyond the tensors themselves: a host that
 * owns all device memory through its own allocator and gives plugins only
 * inputs and outputs, or a steady-state decode loop that must not call
 * cudaMalloc (it can synchronise the whole device) between tokens.  There is
 * no counterpart on the pages; this is an interface convenience only.
 *
 * Arguments, layouts, math and results are those of attn_decode_gqa.  The
 * split partials and arrival counters live in a 4 MiB array that is part of
 * the library's device image: every GPU that loads the library holds it until
 * the process exits.  Nothing is allocated per call.
 *   - Limit: the call needs about B*Hkv*splits*G'*(D+2)*4 bytes (G' = Hq/Hkv
 *     rounded up to a power of two; splits <= 3*SMs/(B*Hkv), at least 1); a
 *     problem that does not fit the 4 MiB returns ATTN_ERR_RESOURCE.
 *   - Every call on a device shares the array and leaves its contents behind;
 *     each call zeroes the counters it uses first.  Calls that may overlap on
 *     the GPU (other streams, other host threads) race: serialise them.
 *   - The first call on a device looks up the array's device address; make
 *     that first call outside any stream capture.
 *   - `stream` must belong to the current device (the array used is the
 *     current device's); a stream of another device returns
 *     ATTN_ERR_INVALID_ARG and launches nothing.
 */
ATTN_API attn_status_t attn_decode_gqa_noalloc(const void *q, const void *k_cache,
                                               const void *v_cache, const int32_t *seq_len,
                                               void *o, int B, int Hq, int Hkv, int Lmax, int D,
                                               attn_dtype_t dtype, float scale, void *stream);

/*
 * Appends one token's K and V rows to a KV cache at the position the device
 * holds, for a decode step that is captured once as a CUDA graph and replayed
 * per token with unchanged arguments.
 *   k_cache, v_cache [B, Hkv, Lmax, D] (written: row seq_len[b] of every KV
 *   head of batch b); k_new, v_new [B, Hkv, D] (read).  seq_len: DEVICE int32
 *   [B], the write position; if advance != 0 the kernel then sets
 *   seq_len[b] += 1 (so a following attn_decode_gqa sees the new token).
 *   A position outside [0, Lmax) writes nothing and sets ATTN_ERR_DEVICE_CHECK.
 *   dtype ATTN_F32, ATTN_BF16 or ATTN_F16; D in {32, 64, 128}.
 * Passage: fak "GPU - the in-kernel forward pass", section 3b, step 3 (a
 * kernel-form KV append with a scalar offset replaces the cudaMemcpy whose
 * moving destination forced a graph re-instantiation every token).
 */
ATTN_API attn_status_t attn_kv_append(void *k_cache, void *v_cache, const void *k_new,
                                      const void *v_new, int32_t *seq_len, int B, int Hkv,
                                      int Lmax, int D, attn_dtype_t dtype, int advance,
                                      void *stream);

/*
 * Ring KV cache: the pair attn_kv_append_ring / attn_decode_gqa_ring keeps the
 * most recent Lmax tokens of a sequence in a cache of Lmax rows, so a decode
 * loop captured once as a CUDA graph runs past the cache capacity instead of
 * stopping at it (a sliding attention window of Lmax tokens).
 *   seq_len[b] counts every token appended to sequence b so far (it may
 *   exceed Lmax); token t lives in row t % Lmax until token t + Lmax
 *   overwrites it.
 *   attn_kv_append_ring: as attn_kv_append, writing row seq_len[b] % Lmax;
 *   seq_len[b] must be >= 0 and below INT32_MAX, else nothing is written and
 *   ATTN_ERR_DEVICE_CHECK is set.
 *   attn_decode_gqa_ring: as attn_decode_gqa, attending to the
 *   min(seq_len[b], Lmax) rows that hold tokens, i.e. to tokens
 *   [seq_len[b] - Lmax, seq_len[b]) once the ring has wrapped; seq_len[b] >= 1
 *   with no upper bound.  The row order does not change the result: the
 *   softmax-weighted sum runs over a set of keys, whose positions are already
 *   in their rotated K rows.  Same workspace contract as attn_decode_gqa.
 * Passage: fak "GPU - the in-kernel forward pass", section 3b (the device KV
 * of fixed capacity, with a dynamic / ring device KV named as the follow-up).
 * With Lmax a call argument, a larger capacity is a new cache and a new
 * capture; the ring is what lets one capture run indefinitely.
 */
ATTN_API attn_status_t attn_kv_append_ring(void *k_cache, void *v_cache, const void *k_new,
                                           const void *v_new, int32_t *seq_len, int B, int Hkv,
                                           int Lmax, int D, attn_dtype_t dtype, int advance,
                                           void *stream);
ATTN_API attn_status_t attn_decode_gqa_ring(const void *q, const void *k_cache,
                                            const void *v_cache, const int32_t *seq_len,
                                            void *o, int B, int Hq, int Hkv, int Lmax, int D,
                                            attn_dtype_t dtype, float scale, void *workspace,
                                            size_t workspace_bytes, void *stream);

/*
 * 3D neighborhood attention with NATTEN boundary windows.
 *   q, k, v, o [B, heads, N, D] with N = T * Hg * W tokens in row-major
 *   (t, h, w) order.  kernel: HOST int[3], the requested window per axis; each
 *   must be positive and odd, and may exceed the axis extent.  Per axis of
 *   extent n and request k: k_eff = min(k, n); query coordinate i attends to
 *   [s, s + k_eff) with s = clamp(i - k/2, 0, n - k_eff); the 3D window is the
 *   Cartesian product of the three intervals.  A window at least as wide as
 *   its axis is full attention along that axis.
 * Passage: candle PR #11, the "Line-for-line port of neighborhood_attention.metal"
 * commit and the "kernel exceeds grid extent" commit (effective_kernel() clamp,
 * validate() only requires a positive odd triple).
 */
ATTN_API attn_status_t attn_na3d_fwd(const void *q, const void *k, const void *v, void *o,
                            int B, int heads, int T, int Hg, int W, int D,
                            const int kernel[3], attn_dtype_t dtype, float scale,
                            void *stream);

/*
 * 3D neighborhood attention on strided views: the operation of
 * attn_na3d_fwd with q, k, v and o addressed through element strides of
 * (batch, head, token) as in attn_full_fwd_strided (D contiguous, every
 * stride a multiple of 16 bytes, extent-1 axes' strides ignored, o's rows
 * disjoint); tokens keep their row-major (t, h, w) order at a uniform token
 * stride, so a [B, T*Hg*W, heads, D] projection is read in place.  A
 * non-contiguous layout runs on the exact SIMT kernel; contiguous strides
 * take the tensor-core kernel of attn_na3d_fwd.
 * Passage: as attn_na3d_fwd; the layout is an addressing choice with no
 * counterpart in the pages.
 */
ATTN_API attn_status_t attn_na3d_fwd_strided(const void *q, const void *k, const void *v, void *o,
                                            int B, int heads, int T, int Hg, int W, int D,
                                            const int kernel[3], const int64_t q_strides[3],
                                            const int64_t k_strides[3],
                                            const int64_t v_strides[3],
                                            const int64_t o_strides[3], attn_dtype_t dtype,
                                            float scale, void *stream);

/*
 * Window starts as the neighborhood kernels compute them (same device
 * function), for testing: starts = DEVICE int32 [T*Hg*W, 3], the (t, h, w)
 * start of each query's window.  Same validation as attn_na3d_fwd.
 */
ATTN_API attn_status_t attn_na3d_window_starts(int T, int Hg, int W, const int kernel[3],
                                      int32_t *starts, void *stream);

/*
 * Tensor-core building-block check (testing): one CTA computes, for a single
 * tile, S = q k^T + q[:, :16] k[:, :16]^T and O = P v with the same tcgen05
 * MMA forms, shared-memory layouts (128-byte swizzle for q, k, v; 32-byte
 * swizzle for the 16-channel term, as used by the neighborhood kernel's
 * window-penalty channels) and TMEM placement the bf16 attention kernels use.
 *   q, k, v: DEVICE bf16 [128, D]; P: DEVICE bf16 [128, 128];
 *   S: DEVICE f32 [128, 128]; O: DEVICE f32 [128, D]; D in {64, 128}.
 * No counterpart on the pages: it isolates the matrix-descriptor and
 * tensor-memory conventions so a layout error shows up as a wrong tile here.
 */
ATTN_API attn_status_t attn_debug_tc_tile(const void *q, const void *k, const void *v,
                                          const void *P, float *S, float *O, int D,
                                          void *stream);

/*
 * Bounded-wait check (testing): launches one thread that waits on a
 * shared-memory barrier nothing ever completes, with a wait limit of
 * limit_ns nanoseconds (1000 .. 1000000000; outside that range
 * ATTN_ERR_INVALID_ARG and nothing launches).  The wait runs out, sets the
 * device error word to the timeout code and the thread returns, so the
 * next attn_device_status() on this stream returns ATTN_ERR_TIMEOUT (and
 * clears the word) with the context still usable.  Every spin-wait in the
 * attention kernels is this same bounded wait with a limit of one second.
 * No counterpart on the pages: it exercises the library's failure reporting
 * without faulting or hanging a GPU.
 */
ATTN_API attn_status_t attn_debug_wait_test(uint64_t limit_ns, void *stream);

/* Human-readable name of a status code (static storage). */
ATTN_API const char *attn_status_string(attn_status_t status);

/*
 * Synchronises `stream`, then reads and clears the device error word that
 * bounded waits and device-side checks set on the current device.
 * Returns ATTN_OK, ATTN_ERR_TIMEOUT, ATTN_ERR_DEVICE_CHECK or ATTN_ERR_CUDA.
 */
ATTN_API attn_status_t attn_device_status(void *stream);

/*
 * Number of kernel launches this process has made through the given kernel
 * family, for tests that must prove the path under test really ran.
 * ids: 0 = fp32/SIMT flash, 1 = tcgen05 flash, 2 = decode split-KV,
 *      3 = RoPE prologue, 4 = window-start export, 5 = tcgen05 neighborhood,
 *      6 = KV-cache append, 7 = bounded-wait check.
 * Returns 0 for an unknown id.
 */
ATTN_API uint64_t attn_launch_count(int kernel_family);

/* Library version string, e.g. "libattn 0.1 sm_103a". */
ATTN_API const char *attn_version(void);

#ifdef __cplusplus
}
#endif

#endif /* LIBATTN_H */
