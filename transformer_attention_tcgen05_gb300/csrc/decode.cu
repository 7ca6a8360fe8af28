// Split-KV grouped-query decode attention over a bf16 KV cache.
//
// One query token per sequence attends to the first seq_len[b] rows of its
// KV head's cache (fak "GPU - the in-kernel forward pass": device-resident KV
// cache, section 0; the naive one-block-per-head decode attention that
// section 4 lists as a gap).  The work is HBM-bound (4 FLOP per cache byte),
// so the design is about streaming the cache once at full bandwidth with few
// instructions per byte:
//
//  * grid = splits x Hkv x B, sized to about one wave of three CTAs per SM.
//    A CTA owns one contiguous row range of one (batch, kv-head) cache and
//    serves all G = Hq/Hkv query heads of that KV head, so every cache byte is
//    read exactly once (GQA head sharing).
//  * a producer warp streams 32-row chunks of K and V with TMA tensor copies
//    (128-byte swizzle, L2 evict-first) into a 4-slot shared-memory ring;
//    chunk i goes to slot i % 4 and is consumed by consumer warp i % 4.  The
//    K and V halves of a slot have their own barriers and their own producer
//    lane: a warp frees the K half right after Q K^T, so the next chunk's K
//    arrives while it computes P V (with one barrier per slot every warp sat
//    idle for a full load latency per chunk).
//  * Q K^T: lane = cache row.  Each lane reads its row in 16-byte chunks (the
//    swizzle makes the 32 rows' reads bank-conflict free) against q held in
//    shared memory as fp32 (broadcast reads), with packed fp32x2 FMAs.
//  * online softmax per head across the warp's 32 rows (butterfly max), in
//    base 2; P goes to shared memory.
//  * P V: D/8 lanes per row, 8 channels per lane (one 16-byte swizzled read),
//    2 or 4 rows per instruction, packed fp32x2 FMAs.
//  * the CTA merges its warps (log-sum-exp) into one partial (m, l, o) per
//    head.  The splits of a (batch, kv-head) then merge either through
//    distributed shared memory, as one thread-block cluster, or (when the
//    clusters do not all fit on the GPU at once) through the workspace: the
//    last CTA to arrive (atomic ticket) merges all splits and resets its
//    ticket so the workspace is ready for the next call.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <float.h>
#include <math.h>

#include <mutex>

#include "common.cuh"
#include "kernels.h"
#include "ptx.cuh"

namespace attn {
namespace {

constexpr int kRowsPerChunk = 32;
constexpr int kCW = 4;          // consumer warps
constexpr int kSlots = 4;       // ring slots (one chunk each); chunk i -> slot i % kSlots
static_assert(kSlots % kCW == 0, "every slot must always feed the same consumer warp");
constexpr int kMaxSplits = 256;
constexpr int kMaxClusterSplits = 8;   // portable cluster size
constexpr int kFastMergeSplits = 8;    // workspace merge with all split loads in flight at once

template <int D, int GP>
struct DecCfg {
    static constexpr int PANELS = D / 64;
    static constexpr int PANEL = kRowsPerChunk * 128;       // bytes per 64-channel panel
    static constexpr int TILE = PANELS * PANEL;             // K (or V) bytes per chunk
    static constexpr int LPR = D / 8;                       // P V: lanes per row
    static constexpr int RPI = 32 / LPR;                    // P V: rows per instruction
    static constexpr int NT = (kCW + 1) * 32;
    // shared memory (bytes, from a 1024-aligned base)
    static constexpr int OFF_K = 0;
    static constexpr int OFF_V = kSlots * TILE;
    static constexpr int OFF_Q = 2 * kSlots * TILE;                      // [GP][D] f32
    static constexpr int OFF_P = OFF_Q + GP * D * 4;                     // [CW][32][GP] f32
    static constexpr int OFF_BAR = OFF_P + kCW * kRowsPerChunk * GP * 4;
    static constexpr int SMEM = OFF_BAR + 4 * kSlots * 8 + 16 + 1024;
    // the warp-merge area [CW][GP][D+2] f32 reuses the K slots after the loop
    static constexpr int OFF_M = 0;
    // then (cluster merge) the CTA's own partial [GP][D] o and [GP][2] (m, l)
    static constexpr int OFF_CP = OFF_M + kCW * GP * (D + 2) * 4;
    static_assert(OFF_CP + GP * (D + 2) * 4 <= kSlots * TILE,
                  "merge areas must fit the K slots");
};

struct DecParams {
    const void *q;           // [B][Hq][D], bf16 or f16 like the cache
    const int32_t *seq_len;
    void *o;
    int Hq, Hkv, Lmax, G;
    int splits, split_rows, ws_splits;
    int ring;                // seq_len counts every token appended; the cache holds the last Lmax
    float qscale;
    float *part_o;           // [units][ws_splits][GP][D]
    float *part_ml;          // [units][ws_splits][GP][2]
    unsigned *tickets;       // [units]
    unsigned *err;
};

// eight 16-bit values (bf16, or f16 if F16) -> fp32
template <bool F16>
__device__ __forceinline__ void x8_to_f32(const uint4 &u, float (&x)[8]) {
    using H = H16<F16>;
    x[0] = H::lo(u.x); x[1] = H::hi(u.x);
    x[2] = H::lo(u.y); x[3] = H::hi(u.y);
    x[4] = H::lo(u.z); x[5] = H::hi(u.z);
    x[6] = H::lo(u.w); x[7] = H::hi(u.w);
}

// CL: the splits of one (batch, kv-head) form one thread-block cluster and
// merge their partials through distributed shared memory (no workspace, no
// atomics); otherwise the last CTA to arrive merges them from the workspace.
template <int D, int GP, bool CL, bool F16>
__global__ void __launch_bounds__(DecCfg<D, GP>::NT)
decode_kernel(const __grid_constant__ CUtensorMap tk, const __grid_constant__ CUtensorMap tv,
              const DecParams p) {
    using C = DecCfg<D, GP>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024 - (ptx::smem_addr(smem_raw) & 1023)) & 1023);
    // each slot's K and V halves fill and free separately: a warp frees the K
    // half after Q K^T, so the next chunk's K loads while it computes P V
    uint64_t *full_k = reinterpret_cast<uint64_t *>(smem + C::OFF_BAR);
    uint64_t *full_v = full_k + kSlots;
    uint64_t *empty_k = full_v + kSlots;
    uint64_t *empty_v = empty_k + kSlots;
    __shared__ int s_abort;
    __shared__ unsigned s_last;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int split = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;
    const int unit = b * p.Hkv + kvh;

    // launched as a programmatic dependent of the previous kernel on the
    // stream: nothing global is read or written before that kernel has
    // completed (the cache, the lengths or q may be its outputs); the next
    // kernel may start launching at once
    ptx::griddep_wait();
    ptx::griddep_launch_dependents();

    // q of the G heads of this KV head: its loads go out first, before any
    // cache copy of the grid floods the memory system (issued after the
    // barrier set-up, they took ~3.6 us and held up the consumers while the
    // ring sat full)
    constexpr int QL = (GP * D / 8 + kCW * 32 - 1) / (kCW * 32);   // 16-byte loads per consumer thread
    uint4 qraw[QL];
#pragma unroll
    for (int i = 0; i < QL; ++i) {
        qraw[i] = make_uint4(0u, 0u, 0u, 0u);
        const int e = threadIdx.x + i * kCW * 32;
        if (warp < kCW && e < GP * D / 8) {
            const int h = (e * 8) / D, d = (e * 8) % D;
            if (h < p.G)
                qraw[i] = *reinterpret_cast<const uint4 *>(static_cast<const typename H16<F16>::T *>(p.q) +
                                                          (size_t(b) * p.Hq + kvh * p.G + h) * D + d);
        }
    }

    const int len = p.seq_len[b];
    if (len < 1 || (!p.ring && len > p.Lmax)) {   // invalid length: report, touch nothing
        if (threadIdx.x == 0) raise_device_error(p.err, kDevCheck);
        return;
    }
    // rows in use: every row once a ring cache has wrapped (attention over a
    // set of keys does not depend on the order of the rows that hold them)
    const int L = imin(len, p.Lmax);
    const int r0 = split * p.split_rows;
    const int r1 = imin(r0 + p.split_rows, L);
    const int nchunks = r1 > r0 ? cdiv(r1 - r0, kRowsPerChunk) : 0;

    float *q_s = reinterpret_cast<float *>(smem + C::OFF_Q);
    if (threadIdx.x == 0) {
        for (int s = 0; s < 4 * kSlots; ++s) ptx::mbar_init(&full_k[s], 1);
        ptx::fence_barrier_init();
        s_abort = 0;
    }
    __syncthreads();
    if (warp < kCW) {
        // q pre-scaled to fp32 in shared memory (padding heads are zero)
#pragma unroll
        for (int i = 0; i < QL; ++i) {
            const int e = threadIdx.x + i * kCW * 32;
            if (e < GP * D / 8) {
                float x[8];
                x8_to_f32<F16>(qraw[i], x);
#pragma unroll
                for (int c = 0; c < 8; ++c) q_s[e * 8 + c] = x[c] * p.qscale;
            }
        }
        ptx::named_barrier_sync(2, kCW * 32);
    }

    float *s_merge = reinterpret_cast<float *>(smem + C::OFF_M);

    if (warp == kCW) {
        // ------------------------------------------------ producer warp
        // lane 0 streams the K halves of the slots, lane 1 the V halves
        if (lane < 2) {
            const bool is_k = lane == 0;
            const CUtensorMap *tm = is_k ? &tk : &tv;
            uint64_t *fb = is_k ? full_k : full_v;
            uint64_t *eb = is_k ? empty_k : empty_v;
            uint8_t *dst0 = smem + (is_k ? C::OFF_K : C::OFF_V);
            ptx::prefetch_tmap(tm);
            const uint64_t pol = ptx::l2_policy_evict_first();
            int issued = 0;
            for (int it = 0; it < nchunks; ++it) {
                const int s = it % kSlots;
                if (it >= kSlots && !ptx::mbar_wait(&eb[s], ((it / kSlots) - 1) & 1, p.err)) {
                    s_abort = 1;
                    break;
                }
                const int j0 = r0 + it * kRowsPerChunk;
                ptx::mbar_arrive_expect_tx(&fb[s], C::TILE);
                for (int pn = 0; pn < C::PANELS; ++pn)
                    ptx::tma_load_3d(dst0 + s * C::TILE + pn * C::PANEL, tm, pn * 64, j0, unit, &fb[s],
                                     pol);
                issued = it + 1;
            }
            if (s_abort) {
                // let the copies already issued land (bounded) before exiting
                for (int it = imax(0, issued - kSlots); it < issued; ++it)
                    ptx::mbar_wait(&fb[it % kSlots], (it / kSlots) & 1, nullptr);
            }
        }
    } else {
        // ------------------------------------------------ consumer warps
        float m[GP], lrow[GP], acc[GP][8];
#pragma unroll
        for (int h = 0; h < GP; ++h) {
            m[h] = -INFINITY;
            lrow[h] = 0.f;
#pragma unroll
            for (int d = 0; d < 8; ++d) acc[h][d] = 0.f;
        }
        float *p_s = reinterpret_cast<float *>(smem + C::OFF_P) + warp * kRowsPerChunk * GP;
        const int grp = lane / C::LPR;       // P V: row within an instruction
        const int sub = lane % C::LPR;       // P V: channels [8 sub, 8 sub + 8)
        const int vpanel = sub / 8, vchunk = sub % 8;

        for (int it = warp; it < nchunks; it += kCW) {
            const int s = it % kSlots;
            if (!__all_sync(0xffffffffu, ptx::mbar_wait(&full_k[s], (it / kSlots) & 1, p.err))) {
                s_abort = 1;
                break;
            }
            const uint8_t *Kst = smem + C::OFF_K + s * C::TILE;
            const uint8_t *Vst = smem + C::OFF_V + s * C::TILE;
            const int j0 = r0 + it * kRowsPerChunk;
            const int valid = imin(kRowsPerChunk, r1 - j0);

            // ---- scores: lane = cache row
            float sc[GP];
            {
                float a0[GP], a1[GP];
#pragma unroll
                for (int h = 0; h < GP; ++h) a0[h] = a1[h] = 0.f;
                const int r = lane;
#pragma unroll
                for (int c = 0; c < D / 8; ++c) {
                    const int pn = c / 8, cc = c % 8;
                    const uint4 u = *reinterpret_cast<const uint4 *>(
                        Kst + pn * C::PANEL + r * 128 + ((cc ^ (r & 7)) << 4));
                    float kx[8];
                    x8_to_f32<F16>(u, kx);
#pragma unroll
                    for (int h = 0; h < GP; ++h) {
                        const float4 qa = *reinterpret_cast<const float4 *>(q_s + h * D + c * 8);
                        const float4 qb = *reinterpret_cast<const float4 *>(q_s + h * D + c * 8 + 4);
                        ptx::ffma2(a0[h], a1[h], kx[0], kx[1], qa.x, qa.y, a0[h], a1[h]);
                        ptx::ffma2(a0[h], a1[h], kx[2], kx[3], qa.z, qa.w, a0[h], a1[h]);
                        ptx::ffma2(a0[h], a1[h], kx[4], kx[5], qb.x, qb.y, a0[h], a1[h]);
                        ptx::ffma2(a0[h], a1[h], kx[6], kx[7], qb.z, qb.w, a0[h], a1[h]);
                    }
                }
#pragma unroll
                for (int h = 0; h < GP; ++h) sc[h] = (lane < valid) ? a0[h] + a1[h] : -INFINITY;
            }

            // the K half of the slot is free for the chunk kSlots ahead
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(&empty_k[s]);

            // ---- online softmax per head over the warp's 32 rows
            float alpha[GP];
#pragma unroll
            for (int h = 0; h < GP; ++h) {
                float mx = sc[h];
#pragma unroll
                for (int off = 16; off > 0; off >>= 1)
                    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
                const float mn = fmaxf(m[h], mx);
                alpha[h] = (mn == -INFINITY) ? 1.f : ptx::ex2(m[h] - mn);
                const float pr = (mn == -INFINITY) ? 0.f : ptx::ex2(sc[h] - mn);
                m[h] = mn;
                lrow[h] = lrow[h] * alpha[h] + pr;
                p_s[lane * GP + h] = pr;
            }
            __syncwarp();

            if (!__all_sync(0xffffffffu, ptx::mbar_wait(&full_v[s], (it / kSlots) & 1, p.err))) {
                s_abort = 1;
                break;
            }
            // ---- O = O * alpha + P V
#pragma unroll
            for (int h = 0; h < GP; ++h)
#pragma unroll
                for (int d = 0; d < 8; d += 2)
                    ptx::ffma2(acc[h][d], acc[h][d + 1], acc[h][d], acc[h][d + 1], alpha[h], alpha[h],
                               0.f, 0.f);
#pragma unroll 4
            for (int i = 0; i < kRowsPerChunk / C::RPI; ++i) {
                const int r = i * C::RPI + grp;
                if (r < valid) {
                    const uint4 u = *reinterpret_cast<const uint4 *>(
                        Vst + vpanel * C::PANEL + r * 128 + ((vchunk ^ (r & 7)) << 4));
                    float vx[8];
                    x8_to_f32<F16>(u, vx);
                    float pr[GP];
#pragma unroll
                    for (int h = 0; h < GP; ++h) pr[h] = p_s[r * GP + h];
#pragma unroll
                    for (int h = 0; h < GP; ++h)
#pragma unroll
                        for (int d = 0; d < 8; d += 2)
                            ptx::ffma2(acc[h][d], acc[h][d + 1], vx[d], vx[d + 1], pr[h], pr[h],
                                       acc[h][d], acc[h][d + 1]);
                }
            }
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(&empty_v[s]);
        }

        // ---- warp totals: P V over the row groups, row sums over the lanes
#pragma unroll
        for (int h = 0; h < GP; ++h) {
#pragma unroll
            for (int d = 0; d < 8; ++d)
#pragma unroll
                for (int off = C::LPR; off < 32; off <<= 1)
                    acc[h][d] += __shfl_xor_sync(0xffffffffu, acc[h][d], off);
#pragma unroll
            for (int off = 16; off > 0; off >>= 1)
                lrow[h] += __shfl_xor_sync(0xffffffffu, lrow[h], off);
        }
        // every consumer warp is past its last slot read before the merge
        // area (aliasing the K slots) is written
        ptx::named_barrier_sync(1, kCW * 32);
        float *wm = s_merge + warp * GP * (D + 2);
        if (lane < C::LPR) {
#pragma unroll
            for (int h = 0; h < GP; ++h)
#pragma unroll
                for (int d = 0; d < 8; ++d) wm[h * (D + 2) + sub * 8 + d] = acc[h][d];
        }
        if (lane == 0) {
#pragma unroll
            for (int h = 0; h < GP; ++h) {
                wm[h * (D + 2) + D] = m[h];
                wm[h * (D + 2) + D + 1] = lrow[h];
            }
        }
    }
    __syncthreads();

    // ---- CTA merge of the consumer warps -> one partial per head
    const bool aborted = s_abort != 0;
    if constexpr (CL) {
        // Partial into this CTA's shared memory (an aborted CTA's is garbage,
        // the error word is already set); every CTA of the cluster passes both
        // cluster barriers, so none leaves while another reads its memory.
        float *cp_o = reinterpret_cast<float *>(smem + C::OFF_CP);   // [GP][D]
        float *cp_ml = cp_o + GP * D;                                 // [GP][2]
        for (int e = threadIdx.x; e < GP * D; e += C::NT) {
            const int h = e / D, d = e % D;
            float M = -INFINITY;
            for (int w = 0; w < kCW; ++w) M = fmaxf(M, s_merge[(w * GP + h) * (D + 2) + D]);
            float O = 0.f, Lsum = 0.f;
            if (M != -INFINITY) {
                for (int w = 0; w < kCW; ++w) {
                    const float *wm = s_merge + (w * GP + h) * (D + 2);
                    const float f = exp2f(wm[D] - M);   // -inf -> 0
                    O += wm[d] * f;
                    Lsum += wm[D + 1] * f;
                }
            }
            cp_o[e] = O;
            if (d == 0) {
                cp_ml[h * 2] = M;
                cp_ml[h * 2 + 1] = Lsum;
            }
        }
        ptx::cluster_sync();
        // CTA r of the cluster merges heads r, r + splits, ... over all CTAs,
        // in rank order (the same order whichever CTA finishes first)
        const int csz = gridDim.x;               // cluster = the splits of this unit
        const uint32_t o_base = ptx::smem_addr(cp_o), ml_base = ptx::smem_addr(cp_ml);
        for (int h = blockIdx.x; h < p.G; h += csz)
            for (int d = threadIdx.x; d < D; d += C::NT) {
                float ms[kMaxClusterSplits], ls[kMaxClusterSplits], os[kMaxClusterSplits];
                float M = -INFINITY;
#pragma unroll
                for (int r = 0; r < kMaxClusterSplits; ++r) {
                    ms[r] = -INFINITY;
                    ls[r] = os[r] = 0.f;
                    if (r < csz) {
                        ms[r] = ptx::ld_cluster_f32(ptx::cluster_map(ml_base + h * 8, r));
                        ls[r] = ptx::ld_cluster_f32(ptx::cluster_map(ml_base + h * 8 + 4, r));
                        os[r] = ptx::ld_cluster_f32(ptx::cluster_map(o_base + (h * D + d) * 4, r));
                    }
                    M = fmaxf(M, ms[r]);
                }
                float O = 0.f, Lsum = 0.f;
#pragma unroll
                for (int r = 0; r < kMaxClusterSplits; ++r) {
                    const float w = ms[r] == -INFINITY ? 0.f : exp2f(ms[r] - M);
                    O += os[r] * w;
                    Lsum += ls[r] * w;
                }
                static_cast<typename H16<F16>::T *>(p.o)[(size_t(b) * p.Hq + kvh * p.G + h) * D + d] =
                    H16<F16>::from(O / Lsum);
            }
        ptx::cluster_sync();
        return;
    }
    if (!aborted) {
        float *po = p.part_o + (size_t(unit) * p.ws_splits + split) * GP * D;
        float *pml = p.part_ml + (size_t(unit) * p.ws_splits + split) * GP * 2;
        for (int e = threadIdx.x; e < GP * D; e += C::NT) {
            const int h = e / D, d = e % D;
            float M = -INFINITY;
            for (int w = 0; w < kCW; ++w) M = fmaxf(M, s_merge[(w * GP + h) * (D + 2) + D]);
            float O = 0.f, Lsum = 0.f;
            if (M != -INFINITY) {
                for (int w = 0; w < kCW; ++w) {
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

    // ---- last CTA of this (batch, kv-head): merge all splits, write O.
    // Split weights w[s][h] = 2^(m_s - M) / L first (all (m, l) pairs loaded
    // at once into shared memory), then every output element sums its splits
    // with independent loads.
    __threadfence();
    float *wgt = reinterpret_cast<float *>(smem);        // [splits][GP] (slots are free now)
    const float *pml = p.part_ml + size_t(unit) * p.ws_splits * GP * 2;
    const float *po = p.part_o + size_t(unit) * p.ws_splits * GP * D;
    for (int e = threadIdx.x; e < p.splits * GP; e += C::NT) {
        wgt[e * 2] = __ldcg(pml + e * 2);
        wgt[e * 2 + 1] = __ldcg(pml + e * 2 + 1);
    }
    __syncthreads();
    if (threadIdx.x < GP) {
        const int h = threadIdx.x;
        float M = -INFINITY;
        for (int s = 0; s < p.splits; ++s) M = fmaxf(M, wgt[(s * GP + h) * 2]);
        float Lsum = 0.f;
        for (int s = 0; s < p.splits; ++s) {
            const float ms = wgt[(s * GP + h) * 2];
            Lsum += (ms == -INFINITY) ? 0.f : wgt[(s * GP + h) * 2 + 1] * exp2f(ms - M);
        }
        const float inv = 1.f / Lsum;
        for (int s = 0; s < p.splits; ++s) {
            const float ms = wgt[(s * GP + h) * 2];
            wgt[(s * GP + h) * 2 + 1] = (ms == -INFINITY) ? 0.f : exp2f(ms - M) * inv;
        }
    }
    __syncthreads();
    if (p.splits <= kFastMergeSplits) {
        // every partial this thread needs is requested before the first is
        // used (one round trip to L2 instead of one per output and 4 splits)
        constexpr int OPT = (GP * D + C::NT - 1) / C::NT;   // outputs per thread
        float v[OPT][kFastMergeSplits];
#pragma unroll
        for (int k = 0; k < OPT; ++k) {
            const int e = threadIdx.x + k * C::NT, h = e / D, d = e % D;
#pragma unroll
            for (int s = 0; s < kFastMergeSplits; ++s)
                v[k][s] = (e < p.G * D && s < p.splits) ? __ldcg(po + (s * GP + h) * D + d) : 0.f;
        }
#pragma unroll
        for (int k = 0; k < OPT; ++k) {
            const int e = threadIdx.x + k * C::NT, h = e / D, d = e % D;
            if (e < p.G * D) {
                float O = 0.f;
#pragma unroll
                for (int s = 0; s < kFastMergeSplits; ++s)
                    if (s < p.splits) O += v[k][s] * wgt[(s * GP + h) * 2 + 1];
                static_cast<typename H16<F16>::T *>(p.o)[(size_t(b) * p.Hq + kvh * p.G + h) * D + d] =
                    H16<F16>::from(O);
            }
        }
        if (threadIdx.x == 0) p.tickets[unit] = 0u;   // ready for the next call
        return;
    }
    for (int e = threadIdx.x; e < p.G * D; e += C::NT) {
        const int h = e / D, d = e % D;
        float O = 0.f;
        int s = 0;
        for (; s + 4 <= p.splits; s += 4) {
            float v[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) v[i] = __ldcg(po + ((s + i) * GP + h) * D + d);
#pragma unroll
            for (int i = 0; i < 4; ++i) O += v[i] * wgt[((s + i) * GP + h) * 2 + 1];
        }
        for (; s < p.splits; ++s) O += __ldcg(po + (s * GP + h) * D + d) * wgt[(s * GP + h) * 2 + 1];
        static_cast<typename H16<F16>::T *>(p.o)[(size_t(b) * p.Hq + kvh * p.G + h) * D + d] =
            H16<F16>::from(O);
    }
    if (threadIdx.x == 0) p.tickets[unit] = 0u;   // ready for the next call
}

// Largest split count a call can use (sets the workspace layout).
int max_splits_for(int Lmax) {
    return imin(kMaxSplits, imax(1, cdiv(Lmax, kRowsPerChunk) / (2 * kCW)));
}

// CTAs of one configuration that fit an SM (shared memory is the limit).
constexpr int ctas_per_sm(int smem_bytes) {
    return (228 * 1024) / (smem_bytes + 1024) > 0 ? (228 * 1024) / (smem_bytes + 1024) : 1;
}

// Splits per (batch, kv-head): about one wave of resident CTAs, each CTA at
// least two 32-row chunks per consumer warp.
int splits_for(int B, int Hkv, int Lmax, int sm_count) {
    const int units = B * Hkv;
    const int per_sm = ctas_per_sm(DecCfg<128, 4>::SMEM);
    const int splits = imax(1, (per_sm * sm_count) / imax(units, 1));
    return imax(1, imin(splits, max_splits_for(Lmax)));
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn_dec() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
        else
            cudaGetLastError();
    });
    return fn;
}

// 3D map over the cache [units][Lmax][D], box {64, 32, 1}, 128-byte swizzle.
bool cache_tmap(CUtensorMap *m, const void *base, int units, int Lmax, int D, bool f16) {
    auto fn = encode_fn_dec();
    if (!fn) return false;
    const cuuint64_t gdim[3] = {cuuint64_t(D), cuuint64_t(Lmax), cuuint64_t(units)};
    const cuuint64_t gstride[2] = {cuuint64_t(D) * 2, cuuint64_t(Lmax) * D * 2};
    const cuuint32_t box[3] = {64, kRowsPerChunk, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    return fn(m, f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
              const_cast<void *>(base), gdim, gstride, box,
              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int D, int GP, bool F16>
attn_status_t launch(const Ctx &c, const CUtensorMap &tk, const CUtensorMap &tv, DecParams p,
                     int B) {
    using C = DecCfg<D, GP>;
    static int done_mask = 0;
    auto kern = decode_kernel<D, GP, false, F16>;
    if (!ensure_smem_attr(reinterpret_cast<const void *>(kern), C::SMEM, c.device, &done_mask))
        return ATTN_ERR_RESOURCE;
    // programmatic dependent launch: the grid may start (and set up) while
    // the previous kernel finishes; the kernel waits for it before any read
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.splits, p.Hkv, B);
    cfg.blockDim = dim3(C::NT);
    cfg.dynamicSmemBytes = C::SMEM;
    cfg.stream = c.stream;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, kern, tk, tv, p) != cudaSuccess) {
        cudaGetLastError();
        return ATTN_ERR_CUDA;
    }
    return launch_status(kFamDecode);
}

constexpr int kMaxDevices = 64;

// Launch configuration of the cluster-merge kernel: one cluster of `splits`
// CTAs per (batch, kv-head).
template <int D, int GP>
cudaLaunchConfig_t cluster_config(const Ctx &c, int splits, int Hkv, int B,
                                  cudaLaunchAttribute *attr) {
    using C = DecCfg<D, GP>;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(splits, Hkv, B);
    cfg.blockDim = dim3(C::NT);
    cfg.dynamicSmemBytes = C::SMEM;
    cfg.stream = c.stream;
    attr->id = cudaLaunchAttributeClusterDimension;
    attr->val.clusterDim.x = splits;
    attr->val.clusterDim.y = 1;
    attr->val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cfg;
}

// Largest cluster size in [2, min(8, target)] for which the clusters of all
// `units` (batch, kv-head) pairs are resident at once (one wave: no cluster
// waits for another to finish), or 0.  The occupancy answer depends only on
// the device and the kernel, so it is looked up once per size.
template <int D, int GP, bool F16>
int cluster_splits(const Ctx &c, int units, int target) {
    using C = DecCfg<D, GP>;
    static std::mutex mu;
    static int active[kMaxDevices][kMaxClusterSplits + 1];   // 0 = not looked up, -1 = none
    static int done_mask = 0;
    if (c.device < 0 || c.device >= kMaxDevices) return 0;
    auto kern = decode_kernel<D, GP, true, F16>;
    if (!ensure_smem_attr(reinterpret_cast<const void *>(kern), C::SMEM, c.device, &done_mask))
        return 0;
    std::lock_guard<std::mutex> lock(mu);
    for (int cs = imin(kMaxClusterSplits, target); cs >= 2; --cs) {
        int &a = active[c.device][cs];
        if (a == 0) {
            cudaLaunchAttribute attr;
            cudaLaunchConfig_t cfg = cluster_config<D, GP>(c, cs, 1, 1, &attr);
            int n = 0;
            if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) {
                cudaGetLastError();
                n = 0;
            }
            a = n > 0 ? n : -1;
        }
        if (a >= units) return cs;
    }
    return 0;
}

template <int D, int GP, bool F16>
attn_status_t launch_cluster(const Ctx &c, const CUtensorMap &tk, const CUtensorMap &tv,
                             DecParams p, int B) {
    static int done_mask = 0;
    auto kern = decode_kernel<D, GP, true, F16>;
    if (!ensure_smem_attr(reinterpret_cast<const void *>(kern), DecCfg<D, GP>::SMEM, c.device,
                          &done_mask))
        return ATTN_ERR_RESOURCE;
    cudaLaunchAttribute attr[2];
    cudaLaunchConfig_t cfg = cluster_config<D, GP>(c, p.splits, p.Hkv, B, attr);
    // programmatic dependent launch, as for the workspace-merge kernel
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.numAttrs = 2;
    if (cudaLaunchKernelEx(&cfg, kern, tk, tv, p) != cudaSuccess) {
        cudaGetLastError();
        return ATTN_ERR_CUDA;
    }
    return launch_status(kFamDecode);
}

// Cluster merge when every unit's cluster fits one wave, unless the
// workspace (atomic ticket) merge at the call's split count spreads the cache
// over the SMs clearly more evenly: the time of the loop is set by the SM
// with the most CTAs, i.e. by ceil(units x splits / SMs) / splits of a unit.
// (64 units on 152 SMs: clusters of 6 leave SMs with 3 and 2 CTAs of 1/6 of a
// unit each, 7 workspace splits 3 CTAs of 1/7; measured 30.8 vs 30.1 us.)
template <int D, int GP, bool F16>
attn_status_t launch_best(const Ctx &c, const CUtensorMap &tk, const CUtensorMap &tv,
                          DecParams p, int B, int Lmax) {
    const int units = B * p.Hkv;
    const int cs = cluster_splits<D, GP, F16>(c, units, p.splits);
    auto load = [&](int sp) { return double(cdiv(units * sp, imax(1, c.sm_count))) / sp; };
    const bool ws_even =
        cs >= 2 && p.splits <= kFastMergeSplits && p.splits > cs && load(p.splits) < 0.9 * load(cs);
    if (cs >= 2 && !ws_even) {
        p.splits = cs;
        p.split_rows = cdiv(cdiv(Lmax, cs), kRowsPerChunk) * kRowsPerChunk;
        return launch_cluster<D, GP, F16>(c, tk, tv, p, B);
    }
    return launch<D, GP, F16>(c, tk, tv, p, B);
}

// (D, group padding, dtype) dispatch; `best` picks the cluster or the
// workspace merge, otherwise the workspace merge.
template <bool F16>
attn_status_t dispatch(const Ctx &c, const CUtensorMap &tk, const CUtensorMap &tv,
                       const DecParams &p, int B, int Lmax, int D, int GP, bool best) {
    if (D == 128) {
        switch (GP) {
            case 1: return best ? launch_best<128, 1, F16>(c, tk, tv, p, B, Lmax) : launch<128, 1, F16>(c, tk, tv, p, B);
            case 2: return best ? launch_best<128, 2, F16>(c, tk, tv, p, B, Lmax) : launch<128, 2, F16>(c, tk, tv, p, B);
            case 4: return best ? launch_best<128, 4, F16>(c, tk, tv, p, B, Lmax) : launch<128, 4, F16>(c, tk, tv, p, B);
            default: return best ? launch_best<128, 8, F16>(c, tk, tv, p, B, Lmax) : launch<128, 8, F16>(c, tk, tv, p, B);
        }
    }
    switch (GP) {
        case 1: return best ? launch_best<64, 1, F16>(c, tk, tv, p, B, Lmax) : launch<64, 1, F16>(c, tk, tv, p, B);
        case 2: return best ? launch_best<64, 2, F16>(c, tk, tv, p, B, Lmax) : launch<64, 2, F16>(c, tk, tv, p, B);
        case 4: return best ? launch_best<64, 4, F16>(c, tk, tv, p, B, Lmax) : launch<64, 4, F16>(c, tk, tv, p, B);
        default: return best ? launch_best<64, 8, F16>(c, tk, tv, p, B, Lmax) : launch<64, 8, F16>(c, tk, tv, p, B);
    }
}

int gp_for(int G) { return G <= 1 ? 1 : G <= 2 ? 2 : G <= 4 ? 4 : 8; }

}  // namespace

size_t decode_workspace_bytes(int B, int Hq, int Hkv, int Lmax, int D) {
    if (B < 1 || Hkv < 1 || Hq < Hkv || Lmax < 1 || (D != 64 && D != 128)) return 0;
    const int GP = gp_for(Hq / Hkv);
    const int splits = max_splits_for(Lmax);
    const size_t units = size_t(B) * Hkv;
    size_t bytes = units * splits * GP * D * sizeof(float);
    bytes = (bytes + 255) & ~size_t(255);
    bytes += units * splits * GP * 2 * sizeof(float);
    bytes = (bytes + 255) & ~size_t(255);
    bytes += units * sizeof(unsigned);
    return (bytes + 255) & ~size_t(255);
}

attn_status_t decode_gqa(const Ctx &c, attn_dtype_t dt, const void *q, const void *k,
                         const void *v, const int32_t *seq_len, void *o, int B, int Hq, int Hkv,
                         int Lmax, int D, float scale, void *ws, size_t ws_bytes, bool ring) {
    const bool f16 = dt == ATTN_F16;
    const int G = Hq / Hkv;
    const int GP = gp_for(G);
    const size_t need = decode_workspace_bytes(B, Hq, Hkv, Lmax, D);
    if (ws_bytes < need) return ATTN_ERR_RESOURCE;
    if (B > 65535 || Hkv > 65535) return ATTN_ERR_UNSUPPORTED;
    CUtensorMap tk, tv;
    if (!cache_tmap(&tk, k, B * Hkv, Lmax, D, f16) || !cache_tmap(&tv, v, B * Hkv, Lmax, D, f16))
        return ATTN_ERR_CUDA;
    DecParams p{};
    p.q = q;
    p.seq_len = seq_len;
    p.o = o;
    p.Hq = Hq; p.Hkv = Hkv; p.Lmax = Lmax; p.G = G;
    p.ring = ring;
    p.ws_splits = max_splits_for(Lmax);
    p.splits = splits_for(B, Hkv, Lmax, c.sm_count);
    p.split_rows = cdiv(cdiv(Lmax, p.splits), kRowsPerChunk) * kRowsPerChunk;
    p.qscale = scale * kLog2e;
    const size_t units = size_t(B) * Hkv;
    uint8_t *w = static_cast<uint8_t *>(ws);
    size_t off = 0;
    p.part_o = reinterpret_cast<float *>(w + off);
    off = (off + units * p.ws_splits * GP * D * sizeof(float) + 255) & ~size_t(255);
    p.part_ml = reinterpret_cast<float *>(w + off);
    off = (off + units * p.ws_splits * GP * 2 * sizeof(float) + 255) & ~size_t(255);
    p.tickets = reinterpret_cast<unsigned *>(w + off);
    p.err = c.err;
    return f16 ? dispatch<true>(c, tk, tv, p, B, Lmax, D, GP, true)
               : dispatch<false>(c, tk, tv, p, B, Lmax, D, GP, true);
}

// ------------------------------------------------ allocation-free variant
//
// Some callers cannot provide the workspace the split-KV combine needs: a host
// that owns every byte of device memory through its own allocator and hands a
// plugin nothing but input and output tensors, or a steady-state decode loop
// that must not call cudaMalloc (which can synchronise the whole device) between
// tokens.  attn_decode_gqa_noalloc serves them from a fixed scratch array that
// is part of this library's device image: every GPU that loads the library
// holds these kStaticScratchBytes until the process exits, and no call
// allocates anything.
//
// The array is shared by every call on a device and keeps the previous call's
// contents; each call clears the arrival counters it uses before launching.
// Calls that overlap on the GPU (different streams, or several host threads)
// race on the array: serialise them.
//
// The first call on a device looks the array's device address up
// (cudaGetSymbolAddress, with that device current); make that first call
// before any stream capture.

namespace {

constexpr size_t kStaticScratchBytes = size_t(4) << 20;   // 4 MiB per device

__device__ __align__(256) uint8_t g_decode_scratch[kStaticScratchBytes];

constexpr int kMaxScratchDevices = 64;
uint8_t *g_scratch_ptr[kMaxScratchDevices];
std::mutex g_scratch_mu;

// Device address of g_decode_scratch on the current device (looked up once).
attn_status_t scratch_address(int device, uint8_t **out) {
    if (device < 0 || device >= kMaxScratchDevices) return ATTN_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!g_scratch_ptr[device]) {
        void *ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_decode_scratch) != cudaSuccess || ptr == nullptr) {
            cudaGetLastError();
            return ATTN_ERR_CUDA;
        }
        g_scratch_ptr[device] = static_cast<uint8_t *>(ptr);
    }
    *out = g_scratch_ptr[device];
    return ATTN_OK;
}

}  // namespace

}  // namespace attn

extern "C" attn_status_t attn_decode_gqa_noalloc(const void *q, const void *k_cache,
                                                 const void *v_cache, const int32_t *seq_len,
                                                 void *o, int B, int Hq, int Hkv, int Lmax, int D,
                                                 attn_dtype_t dtype, float scale, void *stream) {
    using namespace attn;
    auto a16 = [](const void *ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15u) == 0; };
    if (!q || !k_cache || !v_cache || !seq_len || !o) return ATTN_ERR_INVALID_ARG;
    if (!a16(q) || !a16(k_cache) || !a16(v_cache) || !a16(o)) return ATTN_ERR_INVALID_ARG;
    if (B < 1 || Hq < 1 || Hkv < 1 || Lmax < 1 || Hq % Hkv != 0) return ATTN_ERR_INVALID_ARG;
    if (dtype != ATTN_F32 && dtype != ATTN_BF16 && dtype != ATTN_F16) return ATTN_ERR_INVALID_ARG;
    if (D != 32 && D != 64 && D != 128) return ATTN_ERR_INVALID_ARG;
    if (dtype == ATTN_F32 || D == 32 || Hq / Hkv > 8) return ATTN_ERR_UNSUPPORTED;
    const bool f16 = dtype == ATTN_F16;
    if ((long long)Lmax * D >= (1ll << 31) || B > 65535 || Hkv > 65535) return ATTN_ERR_UNSUPPORTED;
    if (o == q || o == k_cache || o == v_cache) return ATTN_ERR_INVALID_ARG;
    Ctx c;
    attn_status_t st = context_for(stream, &c);
    if (st != ATTN_OK) return st;
    // the scratch address belongs to the current device: a stream of another
    // device would run the kernel against the wrong memory
    if (stream) {
        int sdev = -1;
        if (cudaStreamGetDevice(c.stream, &sdev) != cudaSuccess) {
            cudaGetLastError();
            return ATTN_ERR_INVALID_ARG;
        }
        if (sdev != c.device) return ATTN_ERR_INVALID_ARG;
    }
    uint8_t *scratch = nullptr;
    st = scratch_address(c.device, &scratch);
    if (st != ATTN_OK) return st;

    const int G = Hq / Hkv;
    const int GP = gp_for(G);
    const size_t units = size_t(B) * Hkv;
    DecParams p{};
    p.splits = splits_for(B, Hkv, Lmax, c.sm_count);
    p.ws_splits = p.splits;                     // tight layout: only the splits this call uses
    size_t off_ml = (units * p.splits * GP * D * sizeof(float) + 255) & ~size_t(255);
    size_t off_t = (off_ml + units * p.splits * GP * 2 * sizeof(float) + 255) & ~size_t(255);
    const size_t need = off_t + units * sizeof(unsigned);
    if (need > kStaticScratchBytes) return ATTN_ERR_RESOURCE;   // problem too large for the array

    CUtensorMap tk, tv;
    if (!cache_tmap(&tk, k_cache, B * Hkv, Lmax, D, f16) ||
        !cache_tmap(&tv, v_cache, B * Hkv, Lmax, D, f16))
        return ATTN_ERR_CUDA;
    p.q = q;
    p.seq_len = seq_len;
    p.o = o;
    p.Hq = Hq; p.Hkv = Hkv; p.Lmax = Lmax; p.G = G;
    p.split_rows = cdiv(cdiv(Lmax, p.splits), kRowsPerChunk) * kRowsPerChunk;
    p.qscale = (scale > 0.f && isfinite(scale) ? scale : 1.0f / sqrtf(float(D))) * kLog2e;
    p.part_o = reinterpret_cast<float *>(scratch);
    p.part_ml = reinterpret_cast<float *>(scratch + off_ml);
    p.tickets = reinterpret_cast<unsigned *>(scratch + off_t);
    p.err = c.err;
    // the arrival counters must start at zero whatever the previous call left
    if (cudaMemsetAsync(p.tickets, 0, units * sizeof(unsigned), c.stream) != cudaSuccess) {
        cudaGetLastError();
        return ATTN_ERR_CUDA;
    }
    return f16 ? dispatch<true>(c, tk, tv, p, B, Lmax, D, GP, false)
               : dispatch<false>(c, tk, tv, p, B, Lmax, D, GP, false);
}
