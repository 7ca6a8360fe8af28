// Split-KV grouped-query decode attention over a bf16 KV cache.
//
// One query token per sequence attends to the first seq_len[b] rows of its
// KV head's cache (fak "GPU - the in-kernel forward pass": device-resident KV
// cache, section 0; the naive one-block-per-head decode attention that
// section 4 lists as a gap).  The work is HBM-bound (4 FLOP per cache byte),
// so the design is about streaming the cache once at full bandwidth:
//
//  * grid = splits x Hkv x B.  A CTA owns one contiguous row range of one
//    (batch, kv-head) cache and serves all G = Hq/Hkv query heads of that KV
//    head, so every cache byte is read exactly once (GQA head sharing).
//  * a producer warp streams K and V rows with bulk TMA copies
//    (cp.async.bulk, L2 evict-first) into a 3-stage shared-memory ring
//    guarded by mbarriers; 8 consumer warps compute from shared memory.
//  * consumer lane layout: D/8 lanes per cache row, each lane holding 8
//    channels (one 128-bit shared load per row); a warp covers 32/(D/8) rows
//    per instruction.  Partial dot products of 4 row-instructions x G heads
//    are summed across the row's lanes with a transposing butterfly (each
//    exchange halves the values a lane keeps), then the online softmax runs
//    per head in base 2 and P V accumulates with the same lane layout.
//  * the CTA merges its warps (log-sum-exp) and writes one partial
//    (m, l, o) per head to the workspace; the last CTA of a (batch, kv-head)
//    to arrive (atomic ticket) merges all splits and writes the output, then
//    resets its ticket so the workspace is ready for the next call.
#include <float.h>

#include "common.cuh"
#include "kernels.h"
#include "ptx.cuh"

namespace attn {
namespace {

template <int D, int GP>
struct DecCfg {
    static constexpr int LPR = D / 8;                 // lanes per cache row
    static constexpr int LOG_LPR = (LPR == 16) ? 4 : 3;
    static constexpr int RPI = 32 / LPR;               // rows per warp instruction
    static constexpr int UNR = 4;                      // row-instructions per warp step
    static constexpr int RPW = RPI * UNR;              // rows per warp step
    static constexpr int CW = 8;                       // consumer warps
    static constexpr int NT = (CW + 1) * 32;
    static constexpr int SROWS = RPW * CW;             // rows per stage
    static constexpr int NSTAGE = 3;
    static constexpr int ROWB = D * 2;                 // bytes per cache row
    static constexpr int KBYTES = SROWS * ROWB;        // bytes of K (or V) per stage
    static constexpr int NV = UNR * GP;                // partial scores per lane
    static constexpr int LOG_NV = (NV >= 32) ? 5 : (NV >= 16) ? 4 : (NV >= 8) ? 3 : (NV >= 4) ? 2 : 1;
    static constexpr int NH = LOG_NV < LOG_LPR ? LOG_NV : LOG_LPR;   // halving exchanges
    static constexpr int VPL = NV >> NH;               // values a lane keeps
    static constexpr int SCORES = RPW * GP;            // scores per warp step
    // shared memory carve-up (bytes)
    static constexpr int OFF_K = 0;
    static constexpr int OFF_V = NSTAGE * KBYTES;
    static constexpr int OFF_S = 2 * NSTAGE * KBYTES;                  // [CW][SCORES] f32
    static constexpr int OFF_BAR = OFF_S + CW * SCORES * 4;
    static constexpr int SMEM = OFF_BAR + 2 * NSTAGE * 8 + 16;
    // the warp-merge area [CW][GP][D+2] f32 reuses the K stages after the loop
    static constexpr int OFF_M = 0;
    static_assert(CW * GP * (D + 2) * 4 <= NSTAGE * KBYTES, "merge area must fit the K stages");
    static_assert(NV >= 4, "at least 4 partial scores per lane");
};

struct DecParams {
    const __nv_bfloat16 *q, *k, *v;
    const int32_t *seq_len;
    __nv_bfloat16 *o;
    int Hq, Hkv, Lmax, G;
    int splits, split_rows;
    float qscale;
    float *part_o;           // [units][splits][GP][D]
    float *part_ml;          // [units][splits][GP][2]
    unsigned *tickets;       // [units]
    unsigned *err;
};

template <int VN, int LN>
struct Reduce {
    // Halving butterfly over LN lanes (xor distances LN/2 .. 1, lane bits of
    // `sub`): keeps the upper half of the values where the exchanged bit is
    // set.  When values run out before lanes, the remaining exchanges are
    // plain all-reduce steps.
    static __device__ __forceinline__ void run(float *v, int sub) {
        if constexpr (LN > 1) {
            constexpr int half = LN / 2;
            if constexpr (VN > 1) {
                const bool up = (sub & half) != 0;
#pragma unroll
                for (int j = 0; j < VN / 2; ++j) {
                    const float send = up ? v[j] : v[j + VN / 2];
                    const float keep = up ? v[j + VN / 2] : v[j];
                    v[j] = keep + __shfl_xor_sync(0xffffffffu, send, half);
                }
                Reduce<VN / 2, half>::run(v, sub);
            } else {
                v[0] += __shfl_xor_sync(0xffffffffu, v[0], half);
                Reduce<1, half>::run(v, sub);
            }
        }
    }
};

template <int D, int GP>
__global__ void __launch_bounds__(DecCfg<D, GP>::NT, GP >= 8 ? 1 : 2)
decode_kernel(const DecParams p) {
    using C = DecCfg<D, GP>;
    extern __shared__ __align__(128) uint8_t smem[];
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + C::OFF_BAR);
    uint64_t *empty = full + C::NSTAGE;
    __shared__ int s_abort;
    __shared__ unsigned s_last;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int split = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;
    const int unit = b * p.Hkv + kvh;

    const int L = p.seq_len[b];
    if (L < 1 || L > p.Lmax) {          // invalid length: report, touch nothing
        if (threadIdx.x == 0) raise_device_error(p.err, kDevCheck);
        return;
    }
    const int r0 = split * p.split_rows;
    const int r1 = imin(r0 + p.split_rows, L);
    const int nchunks = r1 > r0 ? cdiv(r1 - r0, C::SROWS) : 0;

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::NSTAGE; ++s) {
            ptx::mbar_init(&full[s], 1);
            ptx::mbar_init(&empty[s], C::CW);
        }
        ptx::fence_barrier_init();
        s_abort = 0;
    }
    __syncthreads();

    const size_t cache_base = (size_t(unit) * p.Lmax) * D;
    float *s_scores = reinterpret_cast<float *>(smem + C::OFF_S);
    float *s_merge = reinterpret_cast<float *>(smem + C::OFF_M);

    if (warp == C::CW) {
        // ------------------------------------------------ producer warp
        if (lane == 0) {
            const uint64_t pol = ptx::l2_policy_evict_first();
            for (int it = 0; it < nchunks; ++it) {
                const int s = it % C::NSTAGE;
                if (it >= C::NSTAGE &&
                    !ptx::mbar_wait(&empty[s], ((it / C::NSTAGE) - 1) & 1, p.err)) {
                    s_abort = 1;
                    break;
                }
                const int j0 = r0 + it * C::SROWS;
                const int rows = imin(C::SROWS, r1 - j0);
                const uint32_t bytes = uint32_t(rows) * C::ROWB;
                ptx::mbar_arrive_expect_tx(&full[s], 2 * bytes);
                ptx::bulk_g2s(smem + C::OFF_K + s * C::KBYTES, p.k + cache_base + size_t(j0) * D,
                              bytes, &full[s], pol);
                ptx::bulk_g2s(smem + C::OFF_V + s * C::KBYTES, p.v + cache_base + size_t(j0) * D,
                              bytes, &full[s], pol);
            }
        }
    } else {
        // ------------------------------------------------ consumer warps
        const int r = lane / C::LPR;       // row within a row-instruction
        const int sub = lane % C::LPR;     // channel group: channels [8 sub, 8 sub + 8)
        float qv[GP][8], acc[GP][8], m[GP];
        float lpart = 0.f;                 // partial row sum of head (lane % GP)
#pragma unroll
        for (int h = 0; h < GP; ++h) {
            m[h] = -INFINITY;
            const int hq = kvh * p.G + h;
            uint4 u = make_uint4(0, 0, 0, 0);
            if (h < p.G)
                u = *reinterpret_cast<const uint4 *>(p.q + (size_t(b) * p.Hq + hq) * D + sub * 8);
            const uint32_t w4[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                qv[h][2 * j] = bf16_lo(w4[j]) * p.qscale;
                qv[h][2 * j + 1] = bf16_hi(w4[j]) * p.qscale;
            }
#pragma unroll
            for (int d = 0; d < 8; ++d) acc[h][d] = 0.f;
        }
        float *sc = s_scores + warp * C::SCORES;

        for (int it = 0; it < nchunks; ++it) {
            const int s = it % C::NSTAGE;
            if (!ptx::mbar_wait(&full[s], (it / C::NSTAGE) & 1, p.err)) {
                s_abort = 1;
                break;
            }
            const uint8_t *Kst = smem + C::OFF_K + s * C::KBYTES;
            const uint8_t *Vst = smem + C::OFF_V + s * C::KBYTES;
            const int j0 = r0 + it * C::SROWS;
            const int wrow0 = warp * C::RPW;               // first stage row of this warp
            const int valid = imin(C::SROWS, r1 - j0) - wrow0;   // rows of this warp in range
            if (valid > 0) {
                // ---- partial scores: UNR row-instructions x GP heads
                float v[C::NV];
#pragma unroll
                for (int i = 0; i < C::UNR; ++i) {
                    const int row = wrow0 + i * C::RPI + r;
                    const uint4 u = *reinterpret_cast<const uint4 *>(Kst + row * C::ROWB + sub * 16);
                    const uint32_t w4[4] = {u.x, u.y, u.z, u.w};
                    float kx[8];
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        kx[2 * j] = bf16_lo(w4[j]);
                        kx[2 * j + 1] = bf16_hi(w4[j]);
                    }
#pragma unroll
                    for (int h = 0; h < GP; ++h) {
                        float a = 0.f;
#pragma unroll
                        for (int d = 0; d < 8; ++d) a = fmaf(qv[h][d], kx[d], a);
                        v[i * GP + h] = a;
                    }
                }
                Reduce<C::NV, C::LPR>::run(v, sub);
                // lane keeps flat indices f = blk * VPL + j (f = i * GP + h)
                const int blk = sub >> (C::LOG_LPR - C::NH);
#pragma unroll
                for (int j = 0; j < C::VPL; ++j) {
                    const int f = blk * C::VPL + j;
                    const int i = f / GP, h = f % GP;
                    const int wr = i * C::RPI + r;         // row within the warp step
                    sc[wr * GP + h] = (wr < valid) ? v[j] : -INFINITY;
                }
                __syncwarp();
                // ---- per-head maximum of this step and the rescale factors
                float mx = -INFINITY;
#pragma unroll
                for (int e = lane; e < C::SCORES; e += 32) mx = fmaxf(mx, sc[e]);
#pragma unroll
                for (int off = GP; off < 32; off <<= 1)
                    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
                float alpha[GP];
#pragma unroll
                for (int h = 0; h < GP; ++h) {
                    const float mh = __shfl_sync(0xffffffffu, mx, h);
                    const float mn = fmaxf(m[h], mh);
                    alpha[h] = (mn == -INFINITY) ? 1.f : exp2f(m[h] - mn);
                    m[h] = mn;
                }
                // ---- probabilities (in place) and the lane's row-sum share
                const int myh = lane % GP;
                float mine = m[0];
#pragma unroll
                for (int h = 1; h < GP; ++h)
                    if (myh == h) mine = m[h];
                float ps = 0.f;
#pragma unroll
                for (int e = lane; e < C::SCORES; e += 32) {
                    const float pe = (mine == -INFINITY) ? 0.f : exp2f(sc[e] - mine);
                    sc[e] = pe;
                    ps += pe;
                }
                float amine = alpha[0];
#pragma unroll
                for (int h = 1; h < GP; ++h)
                    if (myh == h) amine = alpha[h];
                lpart = lpart * amine + ps;
                __syncwarp();
                // ---- O = O * alpha + P V
#pragma unroll
                for (int h = 0; h < GP; ++h)
#pragma unroll
                    for (int d = 0; d < 8; ++d) acc[h][d] *= alpha[h];
#pragma unroll
                for (int i = 0; i < C::UNR; ++i) {
                    const int wr = i * C::RPI + r;
                    if (wr < valid) {
                        const uint4 u =
                            *reinterpret_cast<const uint4 *>(Vst + (wrow0 + wr) * C::ROWB + sub * 16);
                        const uint32_t w4[4] = {u.x, u.y, u.z, u.w};
                        float vx[8];
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            vx[2 * j] = bf16_lo(w4[j]);
                            vx[2 * j + 1] = bf16_hi(w4[j]);
                        }
                        float pr[GP];
#pragma unroll
                        for (int h = 0; h < GP; ++h) pr[h] = sc[wr * GP + h];
#pragma unroll
                        for (int h = 0; h < GP; ++h)
#pragma unroll
                            for (int d = 0; d < 8; ++d) acc[h][d] = fmaf(pr[h], vx[d], acc[h][d]);
                    }
                }
                __syncwarp();
            }
            if (lane == 0) ptx::mbar_arrive(&empty[s]);
        }

        // ---- warp totals: sum the row groups (lanes with equal `sub`)
#pragma unroll
        for (int h = 0; h < GP; ++h)
#pragma unroll
            for (int d = 0; d < 8; ++d)
#pragma unroll
                for (int off = C::LPR; off < 32; off <<= 1)
                    acc[h][d] += __shfl_xor_sync(0xffffffffu, acc[h][d], off);
        // row sums: lanes with equal (lane % GP) hold shares of one head
#pragma unroll
        for (int off = GP; off < 32; off <<= 1) lpart += __shfl_xor_sync(0xffffffffu, lpart, off);
        // every consumer warp is past its last stage read before the merge
        // area (aliasing the K stages) is written
        ptx::named_barrier_sync(1, C::CW * 32);
        float *wm = s_merge + warp * GP * (D + 2);
        if (lane < C::LPR) {
#pragma unroll
            for (int h = 0; h < GP; ++h)
#pragma unroll
                for (int d = 0; d < 8; ++d) wm[h * (D + 2) + sub * 8 + d] = acc[h][d];
        }
        if (lane < GP) {
            wm[lane * (D + 2) + D] = m[lane];
            wm[lane * (D + 2) + D + 1] = lpart;
        }
    }
    __syncthreads();

    // ---- CTA merge of the consumer warps -> one partial per head
    const bool aborted = s_abort != 0;
    if (!aborted) {
        float *po = p.part_o + (size_t(unit) * p.splits + split) * GP * D;
        float *pml = p.part_ml + (size_t(unit) * p.splits + split) * GP * 2;
        for (int e = threadIdx.x; e < GP * D; e += C::NT) {
            const int h = e / D, d = e % D;
            float M = -INFINITY;
            for (int w = 0; w < C::CW; ++w) M = fmaxf(M, s_merge[(w * GP + h) * (D + 2) + D]);
            float O = 0.f, Lsum = 0.f;
            if (M != -INFINITY) {
                for (int w = 0; w < C::CW; ++w) {
                    const float *wm = s_merge + (w * GP + h) * (D + 2);
                    const float f = exp2f(wm[D] - M);   // -inf -> 0
                    O += wm[d] * f;
                    Lsum += wm[D + 1] * f;
                }
            }
            po[e] = O;
            if (d == 0) {
                pml[h * 2] = M;
                pml[h * 2 + 1] = Lsum;
            }
        }
        __threadfence();
    }
    __syncthreads();
    if (aborted) return;
    if (threadIdx.x == 0) {
        const unsigned prev = atomicAdd(&p.tickets[unit], 1u);
        s_last = (prev == unsigned(p.splits) - 1) ? 1u : 0u;
    }
    __syncthreads();
    if (!s_last) return;

    // ---- last CTA of this (batch, kv-head): merge all splits, write O
    __threadfence();
    for (int e = threadIdx.x; e < p.G * D; e += C::NT) {
        const int h = e / D, d = e % D;
        const float *pml = p.part_ml + size_t(unit) * p.splits * GP * 2;
        const float *po = p.part_o + size_t(unit) * p.splits * GP * D;
        float M = -INFINITY;
        for (int s = 0; s < p.splits; ++s) M = fmaxf(M, __ldcg(pml + (s * GP + h) * 2));
        float O = 0.f, Lsum = 0.f;
        for (int s = 0; s < p.splits; ++s) {
            const float ms = __ldcg(pml + (s * GP + h) * 2);
            if (ms == -INFINITY) continue;
            const float f = exp2f(ms - M);
            O += __ldcg(po + (s * GP + h) * D + d) * f;
            Lsum += __ldcg(pml + (s * GP + h) * 2 + 1) * f;
        }
        p.o[(size_t(b) * p.Hq + kvh * p.G + h) * D + d] = __float2bfloat16_rn(O / Lsum);
    }
    if (threadIdx.x == 0) p.tickets[unit] = 0u;   // ready for the next call
}

int splits_for(int B, int Hkv, int Lmax, int srows) {
    const int chunks = cdiv(Lmax, srows);
    // about four stage-chunks per CTA; at least enough CTAs to cover the GPU
    int splits = cdiv(chunks, 4);
    const int units = B * Hkv;
    while (splits < chunks && units * splits < 2 * 152) ++splits;
    return imax(1, imin(splits, 256));
}

template <int D, int GP>
attn_status_t launch(const Ctx &c, DecParams p, int B) {
    using C = DecCfg<D, GP>;
    static int done_mask = 0;
    auto kern = decode_kernel<D, GP>;
    if (!ensure_smem_attr(reinterpret_cast<const void *>(kern), C::SMEM, c.device, &done_mask))
        return ATTN_ERR_RESOURCE;
    kern<<<dim3(p.splits, p.Hkv, B), C::NT, C::SMEM, c.stream>>>(p);
    return launch_status(kFamDecode);
}

int srows_for(int D) { return D == 128 ? DecCfg<128, 4>::SROWS : DecCfg<64, 4>::SROWS; }

int gp_for(int G) { return G <= 1 ? 1 : G <= 2 ? 2 : G <= 4 ? 4 : 8; }

}  // namespace

size_t decode_workspace_bytes(int B, int Hq, int Hkv, int Lmax, int D) {
    if (B < 1 || Hkv < 1 || Hq < Hkv || Lmax < 1 || (D != 64 && D != 128)) return 0;
    const int GP = gp_for(Hq / Hkv);
    const int splits = splits_for(B, Hkv, Lmax, srows_for(D));
    const size_t units = size_t(B) * Hkv;
    size_t bytes = units * splits * GP * D * sizeof(float);
    bytes = (bytes + 255) & ~size_t(255);
    bytes += units * splits * GP * 2 * sizeof(float);
    bytes = (bytes + 255) & ~size_t(255);
    bytes += units * sizeof(unsigned);
    return (bytes + 255) & ~size_t(255);
}

attn_status_t decode_gqa(const Ctx &c, const void *q, const void *k, const void *v,
                         const int32_t *seq_len, void *o, int B, int Hq, int Hkv, int Lmax,
                         int D, float scale, void *ws, size_t ws_bytes) {
    const int G = Hq / Hkv;
    const int GP = gp_for(G);
    const size_t need = decode_workspace_bytes(B, Hq, Hkv, Lmax, D);
    if (ws_bytes < need) return ATTN_ERR_RESOURCE;
    if (B > 65535 || Hkv > 65535) return ATTN_ERR_UNSUPPORTED;
    DecParams p{};
    p.q = static_cast<const __nv_bfloat16 *>(q);
    p.k = static_cast<const __nv_bfloat16 *>(k);
    p.v = static_cast<const __nv_bfloat16 *>(v);
    p.seq_len = seq_len;
    p.o = static_cast<__nv_bfloat16 *>(o);
    p.Hq = Hq; p.Hkv = Hkv; p.Lmax = Lmax; p.G = G;
    const int srows = srows_for(D);
    p.splits = splits_for(B, Hkv, Lmax, srows);
    p.split_rows = cdiv(cdiv(Lmax, p.splits), srows) * srows;
    p.qscale = scale * kLog2e;
    const size_t units = size_t(B) * Hkv;
    uint8_t *w = static_cast<uint8_t *>(ws);
    size_t off = 0;
    p.part_o = reinterpret_cast<float *>(w + off);
    off = (off + units * p.splits * GP * D * sizeof(float) + 255) & ~size_t(255);
    p.part_ml = reinterpret_cast<float *>(w + off);
    off = (off + units * p.splits * GP * 2 * sizeof(float) + 255) & ~size_t(255);
    p.tickets = reinterpret_cast<unsigned *>(w + off);
    p.err = c.err;
    if (D == 128) {
        switch (GP) {
            case 1: return launch<128, 1>(c, p, B);
            case 2: return launch<128, 2>(c, p, B);
            case 4: return launch<128, 4>(c, p, B);
            default: return launch<128, 8>(c, p, B);
        }
    }
    switch (GP) {
        case 1: return launch<64, 1>(c, p, B);
        case 2: return launch<64, 2>(c, p, B);
        case 4: return launch<64, 4>(c, p, B);
        default: return launch<64, 8>(c, p, B);
    }
}

}  // namespace attn
