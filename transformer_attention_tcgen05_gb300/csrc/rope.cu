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
// N/128 query-tile CTAs that read it.  Frequencies come from the host in
// double precision; the angle is one fp32 product, reduced by sincosf.
#include "common.cuh"
#include "kernels.h"

namespace attn {
namespace {

constexpr int kMaxPairs = 64;   // D <= 128

struct RopeParams {
    const void *q, *k;
    void *qr, *kr;
    const int32_t *pos;
    long long total_pairs;       // BH * N * D/2
    int N, Dh;                   // tokens, pairs per row (D/2)
    float freq[kMaxPairs];       // per-pair frequency theta^(-2i/n_a)
    int8_t axis[kMaxPairs];      // per-pair axis index
};

template <typename T>
__global__ void __launch_bounds__(256) rope_kernel(const RopeParams p) {
    for (long long e = blockIdx.x * 256ll + threadIdx.x; e < p.total_pairs;
         e += 256ll * gridDim.x) {
        const int pair = int(e % p.Dh);
        const long long row = e / p.Dh;           // (bh, t)
        const int t = int(row % p.N);
        const float ang = float(p.pos[t * 4 + p.axis[pair]]) * p.freq[pair];
        float sn, cs;
        sincosf(ang, &sn, &cs);
        const size_t off = size_t(e) * 2;
        const T *src[2] = {static_cast<const T *>(p.q), static_cast<const T *>(p.k)};
        T *dst[2] = {static_cast<T *>(p.qr), static_cast<T *>(p.kr)};
#pragma unroll
        for (int w = 0; w < 2; ++w) {
            const float x0 = Elem<T>::load(src[w] + off);
            const float x1 = Elem<T>::load(src[w] + off + 1);
            Elem<T>::store(dst[w] + off, x0 * cs - x1 * sn);
            Elem<T>::store(dst[w] + off + 1, x0 * sn + x1 * cs);
        }
    }
}

}  // namespace

attn_status_t rope_rotate_qk(const Ctx &c, attn_dtype_t dt, const void *q, const void *k,
                             void *qr, void *kr, int BH, int N, int D, const int32_t *pos,
                             const int axes_dim[4], float theta) {
    RopeParams p{};
    p.q = q; p.k = k; p.qr = qr; p.kr = kr; p.pos = pos;
    p.N = N;
    p.Dh = D / 2;
    p.total_pairs = (long long)BH * N * (D / 2);
    int ch = 0;
    for (int a = 0; a < 4; ++a) {
        for (int i = 0; i < axes_dim[a] / 2; ++i) {
            const int pr = ch / 2 + i;
            p.freq[pr] = float(pow(double(theta), -2.0 * i / double(axes_dim[a])));
            p.axis[pr] = int8_t(a);
        }
        ch += axes_dim[a];
    }
    long long blocks = (p.total_pairs + 255) / 256;
    if (blocks > 32ll * c.sm_count) blocks = 32ll * c.sm_count;
    if (blocks < 1) blocks = 1;
    if (dt == ATTN_F32)
        rope_kernel<float><<<int(blocks), 256, 0, c.stream>>>(p);
    else
        rope_kernel<__nv_bfloat16><<<int(blocks), 256, 0, c.stream>>>(p);
    return launch_status(kFamRope);
}

}  // namespace attn
