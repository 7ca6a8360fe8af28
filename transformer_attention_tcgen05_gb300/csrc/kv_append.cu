// Kernel-form KV-cache append for a graph-stable decode step.
//
// fak "GPU - the in-kernel forward pass", section 3b (step 3): a decode loop
// can replay one captured CUDA graph per token only if no node's arguments
// move between tokens; the KV append therefore has to be a kernel that reads
// its write position from device memory (a scalar offset) instead of a
// cudaMemcpy whose destination pointer grows every token.  Here the write
// position of batch b is seq_len[b] itself, read on the device; after writing
// row seq_len[b] of every KV head the kernel (optionally) advances seq_len[b]
// by one, so the same launch -- and the decode launch after it, which reads
// the new length -- can be replayed token after token with unchanged
// arguments.
//
// One CTA per batch row reads its length once, copies the new K and V rows of
// all KV heads with 16-byte vector stores, and only then bumps the length, so
// no other CTA ever reads a length this launch changed.
#include "common.cuh"
#include "ptx.cuh"
#include "kernels.h"

namespace attn {
namespace {

template <typename T>
__global__ void __launch_bounds__(128) kv_append_kernel(T *kc, T *vc, const T *kn, const T *vn,
                                                        int32_t *seq_len, int Hkv, int Lmax,
                                                        int D, int advance, int ring,
                                                        unsigned *err) {
    // a decode launched behind this kernel may start setting up at once (it
    // waits for this grid to complete before it reads anything)
    ptx::griddep_launch_dependents();
    const int b = blockIdx.x;
    const int pos = seq_len[b];
    // linear cache: full or corrupt length; ring: a count that cannot advance
    if (pos < 0 || (ring ? pos == 0x7fffffff : pos >= Lmax)) {   // write nothing
        if (threadIdx.x == 0) raise_device_error(err, kDevCheck);
        return;
    }
    const int row = ring ? pos % Lmax : pos;
    constexpr int VEC = 16 / sizeof(T);
    const int per_head = D / VEC;
    for (int i = threadIdx.x; i < Hkv * per_head; i += blockDim.x) {
        const int h = i / per_head, c = i % per_head;
        const size_t src = (size_t(b) * Hkv + h) * D;
        const size_t dst = ((size_t(b) * Hkv + h) * Lmax + row) * D;
        reinterpret_cast<uint4 *>(kc + dst)[c] = reinterpret_cast<const uint4 *>(kn + src)[c];
        reinterpret_cast<uint4 *>(vc + dst)[c] = reinterpret_cast<const uint4 *>(vn + src)[c];
    }
    if (advance) {
        __syncthreads();                      // every thread of this row read `pos`
        if (threadIdx.x == 0) seq_len[b] = pos + 1;
    }
}

}  // namespace

// f16 rows are 2-byte elements like bf16: the same 16-byte copies serve both.
attn_status_t kv_append(const Ctx &c, attn_dtype_t dt, void *kc, void *vc, const void *kn,
                        const void *vn, int32_t *seq_len, int B, int Hkv, int Lmax, int D,
                        int advance, bool ring) {
    if (B > 2147483647) return ATTN_ERR_UNSUPPORTED;
    if (dt == ATTN_F32)
        kv_append_kernel<float><<<B, 128, 0, c.stream>>>(
            static_cast<float *>(kc), static_cast<float *>(vc), static_cast<const float *>(kn),
            static_cast<const float *>(vn), seq_len, Hkv, Lmax, D, advance, ring, c.err);
    else
        kv_append_kernel<__nv_bfloat16><<<B, 128, 0, c.stream>>>(
            static_cast<__nv_bfloat16 *>(kc), static_cast<__nv_bfloat16 *>(vc),
            static_cast<const __nv_bfloat16 *>(kn), static_cast<const __nv_bfloat16 *>(vn), seq_len,
            Hkv, Lmax, D, advance, ring, c.err);
    return launch_status(kFamKvAppend);
}

}  // namespace attn
