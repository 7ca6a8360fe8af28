// SIMT flash attention: exact fp32 FFMA arithmetic (never TF32), online
// softmax in base 2, for full attention and for 3D neighborhood attention.
//
// This is the fp32 path of libattn (the bf16 paths run on the tensor cores).
// The fp32 storage type must not be silently narrowed: candle PR #11's cuDNN
// commits warn that fp32 quietly becoming TF32 moved results from 3.2e-6 to
// 3.3e-4 -- beyond a 1e-4 fp32 tolerance -- so every product here is an FFMA.
//
// Work decomposition: one CTA owns 64 query rows of one (batch, head); each
// row is held by D/32 threads (32 channels each).  Keys stream through shared
// memory in tiles of 64 (converted to fp32).  Neighborhood attention uses the
// "tile union" scheme: a CTA's queries form a 3D box, the keys it loads are
// the union of the box members' clamped windows (a 3D box again, because the
// window start is monotone in the query coordinate), and a per-element test
// masks the keys outside each query's own window.
#include <float.h>

#include "common.cuh"
#include "kernels.h"

namespace attn {
namespace {

constexpr int kRows = 64;    // query rows per CTA
constexpr int kKT = 64;      // keys per shared-memory tile
constexpr int kChunk = 16;   // keys per online-softmax update

struct SimtParams {
    const void *q, *k, *v;
    void *o;
    int Nq, Nkv;
    float qscale;            // scale * log2(e), folded into q
    // neighborhood attention
    int T, Hg, W;
    int kt, kh, kw;          // requested kernel
    int et, eh, ew;          // effective kernel min(k, extent)
    int bt, bh, bw;          // query box
    int nbh, nbw;            // boxes along h and w
    // causal grouped-query prefill (group > 1: KV head = query head / group)
    int causal, group;
    // H query heads: block row bh is batch bh / H, head bh % H; element
    // strides (batch, head, row) of q, k, v, o with D contiguous
    int H;
    TensorStrides sq, sk, sv, so;
};

template <int D>
struct SimtLayout {
    static constexpr int TPR = D / 32;                 // threads per query row
    static constexpr int NT = kRows * TPR;             // threads per CTA
    static constexpr int SLICE = 36;                   // floats per 32-channel slice (+4 pad)
    static constexpr int ROW = TPR * SLICE;            // floats per key row in smem
    static constexpr size_t SMEM = size_t(2) * kKT * ROW * sizeof(float) + kKT * sizeof(int4);
};

template <typename T> __device__ __forceinline__ float4 load4(const T *p);
template <> __device__ __forceinline__ float4 load4<float>(const float *p) {
    return *reinterpret_cast<const float4 *>(p);
}
template <> __device__ __forceinline__ float4 load4<__nv_bfloat16>(const __nv_bfloat16 *p) {
    const uint2 u = *reinterpret_cast<const uint2 *>(p);
    return make_float4(bf16_lo(u.x), bf16_hi(u.x), bf16_lo(u.y), bf16_hi(u.y));
}
template <> __device__ __forceinline__ float4 load4<__half>(const __half *p) {
    const uint2 u = *reinterpret_cast<const uint2 *>(p);
    return make_float4(f16_lo(u.x), f16_hi(u.x), f16_lo(u.y), f16_hi(u.y));
}

template <typename T, int D, bool NA>
__global__ void __launch_bounds__(SimtLayout<D>::NT)
simt_flash_kernel(const SimtParams p) {
    using L = SimtLayout<D>;
    extern __shared__ float4 smem4[];
    float *Ks = reinterpret_cast<float *>(smem4);
    float *Vs = Ks + kKT * L::ROW;
    int4 *kc = reinterpret_cast<int4 *>(Vs + kKT * L::ROW);   // (t, h, w, valid) per tile key

    const int tid = threadIdx.x;
    const int r = tid / L::TPR;
    const int sl = tid % L::TPR;
    const size_t bh = blockIdx.y;
    const int tile = blockIdx.x;

    const long long b = bh / p.H, h = bh % p.H, hk = h / p.group;
    const T *qg = static_cast<const T *>(p.q) + (b * p.sq.b + h * p.sq.h);
    const T *kg = static_cast<const T *>(p.k) + (b * p.sk.b + hk * p.sk.h);
    const T *vg = static_cast<const T *>(p.v) + (b * p.sv.b + hk * p.sv.h);
    T *og = static_cast<T *>(p.o) + (b * p.so.b + h * p.so.h);

    int qi = 0;
    bool qvalid;
    int wst = 0, wsh = 0, wsw = 0;                 // this query's window starts
    int u0t = 0, u0h = 0, u0w = 0, uh = 1, uw = 1;  // union box origin / extents
    int nkeys;
    if (NA) {
        const int nb_hw = p.nbh * p.nbw;
        const int t0 = (tile / nb_hw) * p.bt;
        const int h0 = ((tile / p.nbw) % p.nbh) * p.bh;
        const int w0 = (tile % p.nbw) * p.bw;
        const int dt = r / (p.bh * p.bw), dh = (r / p.bw) % p.bh, dw = r % p.bw;
        const int t = t0 + dt, h = h0 + dh, w = w0 + dw;
        qvalid = r < p.bt * p.bh * p.bw && t < p.T && h < p.Hg && w < p.W;
        if (qvalid) {
            qi = (t * p.Hg + h) * p.W + w;
            wst = na_window_start(t, p.T, p.kt);
            wsh = na_window_start(h, p.Hg, p.kh);
            wsw = na_window_start(w, p.W, p.kw);
        }
        const int t1 = imin(t0 + p.bt, p.T) - 1;
        const int h1 = imin(h0 + p.bh, p.Hg) - 1;
        const int w1 = imin(w0 + p.bw, p.W) - 1;
        u0t = na_window_start(t0, p.T, p.kt);
        u0h = na_window_start(h0, p.Hg, p.kh);
        u0w = na_window_start(w0, p.W, p.kw);
        const int ut = na_window_start(t1, p.T, p.kt) + p.et - u0t;
        uh = na_window_start(h1, p.Hg, p.kh) + p.eh - u0h;
        uw = na_window_start(w1, p.W, p.kw) + p.ew - u0w;
        nkeys = ut * uh * uw;
    } else {
        qi = tile * kRows + r;
        qvalid = qi < p.Nq;
        // causal: keys past the tile's last query are seen by no row of it
        nkeys = p.causal ? imin(p.Nkv, (tile + 1) * kRows) : p.Nkv;
    }

    float qv[32], acc[32];
#pragma unroll
    for (int d = 0; d < 32; d += 4) {
        float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
        if (qvalid) x = load4<T>(qg + qi * p.sq.n + sl * 32 + d);
        qv[d] = x.x * p.qscale;
        qv[d + 1] = x.y * p.qscale;
        qv[d + 2] = x.z * p.qscale;
        qv[d + 3] = x.w * p.qscale;
        acc[d] = acc[d + 1] = acc[d + 2] = acc[d + 3] = 0.f;
    }
    float m = -INFINITY, l = 0.f;

    for (int kb = 0; kb < nkeys; kb += kKT) {
        // ---- stage one key tile (K and V, converted to fp32) in shared memory
        for (int e = tid; e < kKT * D / 4; e += L::NT) {
            const int kk = (e * 4) / D, d0 = (e * 4) % D;
            const int u = kb + kk;
            float4 kx = make_float4(0.f, 0.f, 0.f, 0.f), vx = kx;
            if (u < nkeys) {
                int g;
                if (NA) {
                    const int a = u / (uh * uw), b = (u / uw) % uh, cc = u % uw;
                    const int ta = u0t + a, hb = u0h + b, wc = u0w + cc;
                    g = (ta * p.Hg + hb) * p.W + wc;
                    if (d0 == 0) kc[kk] = make_int4(ta, hb, wc, 1);
                } else {
                    g = u;
                }
                kx = load4<T>(kg + g * p.sk.n + d0);
                vx = load4<T>(vg + g * p.sv.n + d0);
            } else if (d0 == 0) {
                kc[kk] = make_int4(0, 0, 0, 0);
            }
            const int off = kk * L::ROW + (d0 / 32) * L::SLICE + (d0 % 32);
            *reinterpret_cast<float4 *>(Ks + off) = kx;
            *reinterpret_cast<float4 *>(Vs + off) = vx;
        }
        __syncthreads();

        // ---- scores, online softmax and P V over the tile, 16 keys at a time
#pragma unroll 1
        for (int c0 = 0; c0 < kKT; c0 += kChunk) {
            float s[kChunk];
#pragma unroll
            for (int c = 0; c < kChunk; ++c) {
                const float *kr = Ks + (c0 + c) * L::ROW + sl * L::SLICE;
                float part = 0.f;
#pragma unroll
                for (int d = 0; d < 32; d += 4) {
                    const float4 kx = *reinterpret_cast<const float4 *>(kr + d);
                    part = fmaf(qv[d], kx.x, part);
                    part = fmaf(qv[d + 1], kx.y, part);
                    part = fmaf(qv[d + 2], kx.z, part);
                    part = fmaf(qv[d + 3], kx.w, part);
                }
#pragma unroll
                for (int off = 1; off < L::TPR; off <<= 1)
                    part += __shfl_xor_sync(0xffffffffu, part, off);
                bool ok = kb + c0 + c < nkeys;
                if (!NA && p.causal) ok = ok && kb + c0 + c <= qi;
                if (NA) {
                    const int4 kq = kc[c0 + c];
                    ok = ok && unsigned(kq.x - wst) < unsigned(p.et) &&
                         unsigned(kq.y - wsh) < unsigned(p.eh) &&
                         unsigned(kq.z - wsw) < unsigned(p.ew);
                }
                s[c] = ok ? part : -INFINITY;
            }
            float cm = s[0];
#pragma unroll
            for (int c = 1; c < kChunk; ++c) cm = fmaxf(cm, s[c]);
            const float mn = fmaxf(m, cm);
            if (mn != -INFINITY) {
                const float alpha = exp2f(m - mn);   // m == -inf -> 0
                l *= alpha;
#pragma unroll
                for (int d = 0; d < 32; ++d) acc[d] *= alpha;
                m = mn;
#pragma unroll
                for (int c = 0; c < kChunk; ++c) {
                    const float pc = exp2f(s[c] - mn);
                    l += pc;
                    const float *vr = Vs + (c0 + c) * L::ROW + sl * L::SLICE;
#pragma unroll
                    for (int d = 0; d < 32; d += 4) {
                        const float4 vx = *reinterpret_cast<const float4 *>(vr + d);
                        acc[d] = fmaf(pc, vx.x, acc[d]);
                        acc[d + 1] = fmaf(pc, vx.y, acc[d + 1]);
                        acc[d + 2] = fmaf(pc, vx.z, acc[d + 2]);
                        acc[d + 3] = fmaf(pc, vx.w, acc[d + 3]);
                    }
                }
            }
        }
        __syncthreads();
    }

    if (qvalid) {
        const float inv = 1.f / l;
        T *orow = og + qi * p.so.n + sl * 32;
#pragma unroll
        for (int d = 0; d < 32; ++d) Elem<T>::store(orow + d, acc[d] * inv);
    }
}

__global__ void na_starts_kernel(int T, int Hg, int W, int kt, int kh, int kw, int32_t *out) {
    const int64_t n = int64_t(T) * Hg * W;
    for (int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < n;
         i += int64_t(gridDim.x) * blockDim.x) {
        const int t = int(i / (int64_t(Hg) * W));
        const int h = int((i / W) % Hg);
        const int w = int(i % W);
        out[i * 3 + 0] = na_window_start(t, T, kt);
        out[i * 3 + 1] = na_window_start(h, Hg, kh);
        out[i * 3 + 2] = na_window_start(w, W, kw);
    }
}

// Query box (bt, bh, bw), at most `rows` queries, that minimises the number of
// (query, key) pairs the CTAs compute: boxes x union-window size.
void choose_box(int T, int Hg, int W, const int kern[3], int rows, int box[3]) {
    const int ext[3] = {T, Hg, W};
    int64_t best = -1;
    for (int bt = 1; bt <= imin(T, rows); ++bt)
        for (int bh = 1; bh <= imin(Hg, rows / bt); ++bh)
            for (int bw = 1; bw <= imin(W, rows / (bt * bh)); ++bw) {
                const int b[3] = {bt, bh, bw};
                int64_t cost = 1;
                for (int a = 0; a < 3; ++a) {
                    const int keff = imin(kern[a], ext[a]);
                    const int nb = cdiv(ext[a], b[a]);
                    // mean union extent over the boxes of this axis
                    int64_t usum = 0;
                    for (int j = 0; j < nb; ++j) {
                        const int i0 = j * b[a], i1 = imin(i0 + b[a], ext[a]) - 1;
                        usum += na_window_start(i1, ext[a], kern[a]) + keff -
                                na_window_start(i0, ext[a], kern[a]);
                    }
                    cost *= usum;
                }
                if (best < 0 || cost < best) {
                    best = cost;
                    box[0] = bt; box[1] = bh; box[2] = bw;
                }
            }
}

template <typename T, int D, bool NA>
attn_status_t launch(const Ctx &c, const SimtParams &p, int tiles, int BH) {
    using L = SimtLayout<D>;
    static int done_mask = 0;
    auto kern = simt_flash_kernel<T, D, NA>;
    if (!ensure_smem_attr(reinterpret_cast<const void *>(kern), L::SMEM, c.device, &done_mask))
        return ATTN_ERR_RESOURCE;
    if (BH > 65535) return ATTN_ERR_UNSUPPORTED;
    kern<<<dim3(tiles, BH), L::NT, L::SMEM, c.stream>>>(p);
    return launch_status(kFamSimt);
}

template <bool NA>
attn_status_t dispatch(const Ctx &c, attn_dtype_t dt, int D, const SimtParams &p, int tiles,
                       int BH) {
    if (dt == ATTN_F32) {
        if (D == 32) return launch<float, 32, NA>(c, p, tiles, BH);
        if (D == 64) return launch<float, 64, NA>(c, p, tiles, BH);
        if (D == 128) return launch<float, 128, NA>(c, p, tiles, BH);
    } else if (dt == ATTN_F16) {
        if (D == 32) return launch<__half, 32, NA>(c, p, tiles, BH);
        if (D == 64) return launch<__half, 64, NA>(c, p, tiles, BH);
        if (D == 128) return launch<__half, 128, NA>(c, p, tiles, BH);
    } else {
        if (D == 32) return launch<__nv_bfloat16, 32, NA>(c, p, tiles, BH);
        if (D == 64) return launch<__nv_bfloat16, 64, NA>(c, p, tiles, BH);
        if (D == 128) return launch<__nv_bfloat16, 128, NA>(c, p, tiles, BH);
    }
    return ATTN_ERR_UNSUPPORTED;
}

}  // namespace

// Contiguous [B, heads, N, D] strides.
static TensorStrides dense(int heads, int N, int D) {
    return TensorStrides{(long long)heads * N * D, (long long)N * D, D};
}

attn_status_t simt_full(const Ctx &c, attn_dtype_t dt, const void *q, const void *k,
                        const void *v, void *o, int B, int H, int Nq, int Nkv, int D,
                        float scale, const TensorStrides *st) {
    SimtParams p{};
    p.q = q; p.k = k; p.v = v; p.o = o;
    p.Nq = Nq; p.Nkv = Nkv;
    p.qscale = scale * kLog2e;
    p.group = 1;
    p.H = H;
    p.sq = st ? st[0] : dense(H, Nq, D);
    p.sk = st ? st[1] : dense(H, Nkv, D);
    p.sv = st ? st[2] : dense(H, Nkv, D);
    p.so = st ? st[3] : dense(H, Nq, D);
    return dispatch<false>(c, dt, D, p, cdiv(Nq, kRows), B * H);
}

attn_status_t simt_causal_gqa(const Ctx &c, attn_dtype_t dt, const void *q, const void *k,
                              const void *v, void *o, int B, int Hq, int Hkv, int N, int D,
                              float scale, const TensorStrides *st) {
    SimtParams p{};
    p.q = q; p.k = k; p.v = v; p.o = o;
    p.Nq = p.Nkv = N;
    p.qscale = scale * kLog2e;
    p.causal = 1;
    p.group = Hq / Hkv;   // group 1: every head reads its own K/V
    p.H = Hq;
    p.sq = st ? st[0] : dense(Hq, N, D);
    p.sk = st ? st[1] : dense(Hkv, N, D);
    p.sv = st ? st[2] : dense(Hkv, N, D);
    p.so = st ? st[3] : dense(Hq, N, D);
    return dispatch<false>(c, dt, D, p, cdiv(N, kRows), B * Hq);
}

attn_status_t simt_na3d(const Ctx &c, attn_dtype_t dt, const void *q, const void *k,
                        const void *v, void *o, int B, int H, int T, int Hg, int W, int D,
                        const int kernel[3], float scale, const TensorStrides *st) {
    SimtParams p{};
    p.q = q; p.k = k; p.v = v; p.o = o;
    p.Nq = p.Nkv = T * Hg * W;
    p.qscale = scale * kLog2e;
    p.group = 1;
    p.H = H;
    p.sq = st ? st[0] : dense(H, p.Nq, D);
    p.sk = st ? st[1] : dense(H, p.Nq, D);
    p.sv = st ? st[2] : dense(H, p.Nq, D);
    p.so = st ? st[3] : dense(H, p.Nq, D);
    p.T = T; p.Hg = Hg; p.W = W;
    p.kt = kernel[0]; p.kh = kernel[1]; p.kw = kernel[2];
    p.et = imin(kernel[0], T); p.eh = imin(kernel[1], Hg); p.ew = imin(kernel[2], W);
    int box[3];
    choose_box(T, Hg, W, kernel, kRows, box);
    p.bt = box[0]; p.bh = box[1]; p.bw = box[2];
    p.nbh = cdiv(Hg, p.bh);
    p.nbw = cdiv(W, p.bw);
    const int tiles = cdiv(T, p.bt) * p.nbh * p.nbw;
    return dispatch<true>(c, dt, D, p, tiles, B * H);
}

attn_status_t na_starts(const Ctx &c, int T, int Hg, int W, const int kernel[3],
                        int32_t *starts) {
    const int64_t n = int64_t(T) * Hg * W;
    const int blocks = int((n + 255) / 256 < 4096 ? (n + 255) / 256 : 4096);
    na_starts_kernel<<<blocks, 256, 0, c.stream>>>(T, Hg, W, kernel[0], kernel[1], kernel[2],
                                                   starts);
    return launch_status(kFamNaStarts);
}

}  // namespace attn
