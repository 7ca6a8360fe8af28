// RoPE prologue of the joint text+image path: rotated copies of Q and K.
//
// FLUX's multi-axis rotary embedding (iris.c issue #15 "CUDA codepath !",
// GGML lessons item 3: 4 axes [32,32,32,32], separate text/image positions,
// repeat_interleave): the D channels are cut into 4 consecutive axis blocks;
// inside the block of axis a (width n_a) the adjacent pair (2i, 2i+1) turns by
//     phi = pos[t][a] * theta^(-2i / n_a)
//     x0' = x0 cos(phi) - x1 sin(phi),  x1' = x0 sin(phi) + x1 cos(phi).
//
// One pass over Q and K (HBM-bound: read 2, write 2 tensors) leaves the
// rotated copies in the caller's workspace, so the attention kernel streams
// pre-rotated K tiles instead of re-rotating every K tile in each of the
// N/128 query-tile CTAs that read it.
//
// Layout of the work: a thread owns 8 consecutive channels (4 pairs, one
// 16-byte load for bf16) of one token row and applies them to the same row
// of every head, so cos/sin of a (token, pair) is computed once per CTA column
// instead of once per head.  Frequencies come from the host in double
// precision; the angle is one fp32 product, reduced by sincosf.
#include "common.cuh"
#include "ptx.cuh"
#include "kernels.h"

namespace attn {
namespace {

constexpr int kMaxPairs = 64;   // D <= 128

struct RopeParams {
    const void *q, *k;
    void *qr, *kr;
    const int32_t *pos;
    int BH, N, D;
    float freq[kMaxPairs];       // per-pair frequency theta^(-2i/n_a)
    int8_t axis[kMaxPairs];      // per-pair axis index
};

template <typename T> struct Vec8;
// eight 16-bit values (bf16 or f16) in one 16-byte vector
template <bool F16> struct Vec8H {
    uint4 u;
    __device__ __forceinline__ void load(const void *p) { u = *reinterpret_cast<const uint4 *>(p); }
    __device__ __forceinline__ void store(void *p) const { *reinterpret_cast<uint4 *>(p) = u; }
    __device__ __forceinline__ float get(int i) const {
        const uint32_t w = i < 2 ? u.x : i < 4 ? u.y : i < 6 ? u.z : u.w;
        return (i & 1) ? H16<F16>::hi(w) : H16<F16>::lo(w);
    }
    __device__ __forceinline__ void set2(int pr, float a, float b) {
        const uint32_t w = H16<F16>::pack(a, b);
        if (pr == 0) u.x = w; else if (pr == 1) u.y = w; else if (pr == 2) u.z = w; else u.w = w;
    }
};
template <> struct Vec8<__nv_bfloat16> : Vec8H<false> {};
template <> struct Vec8<__half> : Vec8H<true> {};
template <> struct Vec8<float> {
    float4 a, b;
    __device__ __forceinline__ void load(const void *p) {
        a = reinterpret_cast<const float4 *>(p)[0];
        b = reinterpret_cast<const float4 *>(p)[1];
    }
    __device__ __forceinline__ void store(void *p) const {
        reinterpret_cast<float4 *>(p)[0] = a;
        reinterpret_cast<float4 *>(p)[1] = b;
    }
    __device__ __forceinline__ float get(int i) const {
        const float v[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
        return v[i];
    }
    __device__ __forceinline__ void set2(int pr, float x, float y) {
        if (pr == 0) { a.x = x; a.y = y; } else if (pr == 1) { a.z = x; a.w = y; }
        else if (pr == 2) { b.x = x; b.y = y; } else { b.z = x; b.w = y; }
    }
};

// grid: (ceil(N * D/8 / 256), ceil(BH / heads_per_cta)); thread -> (token, 8-channel group)
template <typename T>
__global__ void __launch_bounds__(256) rope_kernel(const RopeParams p, int heads_per_cta) {
    // the attention kernel behind this pass may start setting up at once (it
    // waits for this grid to complete before it reads the rotated copies)
    ptx::griddep_launch_dependents();
    const int groups = p.D / 8;
    const long long e = blockIdx.x * 256ll + threadIdx.x;
    if (e >= (long long)p.N * groups) return;
    const int t = int(e / groups), g = int(e % groups);
    const int h0 = blockIdx.y * heads_per_cta, h1 = imin(h0 + heads_per_cta, p.BH);
    const T *src[2] = {static_cast<const T *>(p.q), static_cast<const T *>(p.k)};
    T *dst[2] = {static_cast<T *>(p.qr), static_cast<T *>(p.kr)};
    // kBatch heads at a time, every load of the batch issued before the first
    // store, so 2 * kBatch 16-byte loads per thread are in flight at once; the
    // first batch's loads go out before the angles are computed, so the
    // sincos work overlaps them instead of delaying them
    constexpr int kBatch = 4;
    float cs[4], sn[4];
    bool have_angles = false;
    for (int hb = h0; hb < h1; hb += kBatch) {
        Vec8<T> x[2][kBatch];
#pragma unroll
        for (int b = 0; b < kBatch; ++b)
            if (hb + b < h1) {
                const size_t off = (size_t(hb + b) * p.N + t) * p.D + g * 8;
                x[0][b].load(src[0] + off);
                x[1][b].load(src[1] + off);
            }
        if (!have_angles) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int pr = g * 4 + i;
                const float ang = float(p.pos[t * 4 + p.axis[pr]]) * p.freq[pr];
                sincosf(ang, &sn[i], &cs[i]);
            }
            have_angles = true;
        }
#pragma unroll
        for (int b = 0; b < kBatch; ++b)
            if (hb + b < h1) {
                const size_t off = (size_t(hb + b) * p.N + t) * p.D + g * 8;
#pragma unroll
                for (int w = 0; w < 2; ++w) {
                    Vec8<T> y = x[w][b];
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const float x0 = x[w][b].get(2 * i), x1 = x[w][b].get(2 * i + 1);
                        y.set2(i, x0 * cs[i] - x1 * sn[i], x0 * sn[i] + x1 * cs[i]);
                    }
                    y.store(dst[w] + off);
                }
            }
    }
}

}  // namespace

attn_status_t rope_rotate_qk(const Ctx &c, attn_dtype_t dt, const void *q, const void *k,
                             void *qr, void *kr, int BH, int N, int D, const int32_t *pos,
                             const int axes_dim[4], float theta) {
    RopeParams p{};
    p.q = q; p.k = k; p.qr = qr; p.kr = kr; p.pos = pos;
    p.BH = BH; p.N = N; p.D = D;
    int ch = 0;
    for (int a = 0; a < 4; ++a) {
        for (int i = 0; i < axes_dim[a] / 2; ++i) {
            const int pr = ch / 2 + i;
            p.freq[pr] = float(pow(double(theta), -2.0 * i / double(axes_dim[a])));
            p.axis[pr] = int8_t(a);
        }
        ch += axes_dim[a];
    }
    // enough CTAs to fill the GPU several times over; each reuses its
    // cos/sin across `heads_per_cta` heads
    const long long cols = ((long long)N * (D / 8) + 255) / 256;
    int hpc = 1;
    while (hpc < BH && cols * cdiv(BH, hpc * 2) >= 8ll * c.sm_count) hpc *= 2;
    const dim3 grid(unsigned(cols), unsigned(cdiv(BH, hpc)));
    if (dt == ATTN_F32)
        rope_kernel<float><<<grid, 256, 0, c.stream>>>(p, hpc);
    else if (dt == ATTN_F16)
        rope_kernel<__half><<<grid, 256, 0, c.stream>>>(p, hpc);
    else
        rope_kernel<__nv_bfloat16><<<grid, 256, 0, c.stream>>>(p, hpc);
    return launch_status(kFamRope);
}

}  // namespace attn
