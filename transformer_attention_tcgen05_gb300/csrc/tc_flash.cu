// Tensor-core (tcgen05 + TMEM + TMA) flash attention for bf16 and f16, sm_103a.
//
// S = Q K^T * scale, row softmax, O = P V, streamed over key tiles with an
// online softmax (the attention of iris.c issue #15 "CUDA codepath !" and the
// neighborhood attention of candle PR #11).  The pages compute it as cuBLAS
// GEMM -> softmax kernel -> GEMM with S in HBM, or as a one-block-per-query
// SIMT kernel; here S and P never leave the SM.
//
// One CTA = two 128-row query tiles (Q0, Q1) of one (batch, head), 12 warps:
//   warps 0-3   softmax warpgroup of Q0 (thread = query row = TMEM lane)
//   warps 4-7   softmax warpgroup of Q1
//   warp  8     MMA issuer (one elected thread) and TMEM owner
//   warp  9     TMA loader of Q and K (one elected thread)
//   warp 10     TMA loader of V (one elected thread); warp 11 only donates
//               registers: the third warpgroup drops to 72 registers per
//               thread (setmaxnreg) so the softmax warpgroups can hold a whole
//               128-column S row in registers (216 per thread).
// Tensor memory (512 columns): S_t at [128 t, 128 t + 128), O_t at
// [256 + D t, 256 + D (t + 1)).  With D = 128 the columns are full and P_t
// (bf16, two per column) overwrites the first 64 columns of S_t once the
// softmax has read S_t; with D = 64 P_t has columns of its own
// ([384 + 64 t, 448 + 64 t)).  The P V MMA takes P straight from TMEM
// (A operand) and V from shared memory (MN-major B operand).
//
// Issue order of the MMA thread per key tile j:
//   D = 128 (P over S):  PV0(j), QK0(j+1), PV1(j), QK1(j+1)   -- QK_t(j+1)
//       overwrites S_t only after PV_t(j) has read P_t (MMAs of one thread
//       execute in issue order), so each softmax warpgroup hides behind the
//       other tile's PV and QK;
//   D = 64 (separate P): QK0(j+1), QK1(j+1) as soon as the softmax has read
//       S_t(j) into registers, then PV0(j), PV1(j) -- the next S is computed
//       while the softmax of the current tile runs.
//
// Softmax (base 2): x = s * scale * log2(e).  The first tile sets the running
// max m; later tiles are exponentiated against m as it stands (no tile-max
// pass) and only a tile whose row sum overflows a bound is redone with its own
// max, which moves m if the tile max exceeds it by more than 8; only then is
// O_t rescaled in TMEM, after waiting for the previous PV_t to complete.
// Every branch that leads to a warp-collective tcgen05.ld / st is uniform
// across the warp.
//
// Full attention: both query tiles share each K/V tile (one stream).  Q, K
// and V are 4D tensor maps {D, N, heads, B} built from each tensor's element
// strides (contiguous for the plain entries), and the epilogue stores through
// the output's strides, so strided views are read and written in place.
// Neighborhood attention: the two query tiles are two 3D boxes adjacent in w;
// each streams the union of its queries' clamped windows as (1, KH, 16)
// (t, h, w) key sub-boxes loaded by 5D TMA.  bf16: the h and w window tests
// enter S as a penalty of -2^100 per violated axis through one extra
// 16-channel MMA k-step (one-hot query offsets against per-sub-box key penalty
// tiles), which drops every masked key exactly (P = 0) for any scores below
// 2^98 in magnitude; f16, whose range cannot hold such a penalty, tests h and
// w per key in the softmax instead.  A key frame outside a row's t window is
// dropped in the softmax (P = 0).
//
// All spin-waits are bounded (1 s); on a timeout the CTA raises the device
// error word, drains what it issued, frees TMEM and exits.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "common.cuh"
#include "kernels.h"
#include "ptx.cuh"

namespace attn {
namespace {

constexpr int kBM = 128;      // query rows per tile (MMA M)
constexpr int kNQ = 2;        // query tiles per CTA
constexpr int kBN = 128;      // max keys per key tile (MMA N of S)
constexpr int kKW = 16;       // neighborhood key sub-box width along w

template <int D, bool NA>
struct TcCfg {
    static constexpr int PANELS = D / 64;                  // 128-byte swizzle panels
    static constexpr int PANEL_Q = kBM * 128;              // bytes per Q panel
    static constexpr int PANEL_KV = kBN * 128;             // bytes per K/V panel
    static constexpr int Q_BYTES = PANELS * PANEL_Q;
    static constexpr int KV_BYTES = PANELS * PANEL_KV;
    static constexpr int STREAMS = NA ? kNQ : 1;           // K/V streams per stage
    // neighborhood window-penalty channels: 16 bf16 per row, 32-byte swizzle.
    // The key-side penalties of a key sub-box depend only on its h and w chunk,
    // so each query box needs at most MAXV distinct penalty tiles, built once.
    static constexpr int X_ROW = 32;
    static constexpr int MAXV = NA ? 6 : 0;
    static constexpr int QX_BYTES = NA ? kNQ * kBM * X_ROW : 0;
    static constexpr int KX_BYTES = kBN * X_ROW;              // one penalty tile
    static constexpr int KXV_BYTES = STREAMS * MAXV * KX_BYTES;
    static constexpr int STAGE_BYTES = 2 * STREAMS * KV_BYTES;
    static constexpr int BUDGET = 227 * 1024 - 2048;
    static constexpr int NS_RAW = (BUDGET - kNQ * Q_BYTES - QX_BYTES - KXV_BYTES) / STAGE_BYTES;
    static constexpr int NSTAGE = NS_RAW > 4 ? 4 : NS_RAW;
    static_assert(NSTAGE >= 2, "at least two K/V stages");
    static constexpr int OFF_Q = 0;
    static constexpr int OFF_QX = kNQ * Q_BYTES;
    static constexpr int OFF_KXV = OFF_QX + QX_BYTES;
    static constexpr int OFF_KV = OFF_KXV + KXV_BYTES;
    static constexpr int OFF_BAR = OFF_KV + NSTAGE * STAGE_BYTES;
    static constexpr int SMEM = OFF_BAR + 512 + 1024;      // barriers + 1024 B alignment slack
    static constexpr uint32_t TM_S = 0;                    // S_t at TM_S + t * kBN
    static constexpr uint32_t TM_O = kNQ * kBN;            // O_t at TM_O + t * D
    static constexpr bool SEP_P = kNQ * (kBN + D + kBN / 2) <= 512;   // P_t has its own columns
    static constexpr uint32_t TM_P = SEP_P ? TM_O + kNQ * D : TM_S;   // P_t at TM_P + t * PSTRIDE
    static constexpr uint32_t PSTRIDE = SEP_P ? kBN / 2 : kBN;
    static constexpr uint32_t TM_COLS = 512;
    static constexpr int NSOFT = 4 * kNQ;
    static constexpr int W_MMA = NSOFT;
    static constexpr int W_LOAD = NSOFT + 1;              // Q and K copies
    static constexpr int W_LOADV = NSOFT + 2;             // V copies
    static constexpr int NT = (NSOFT + 4) * 32;            // 3 warpgroups
    // register split: launch 168 x 384 = 64512; 2 x 128 x 216 + 128 x 72 = 64512
    static constexpr int REGS_LAUNCH = 168;
    static constexpr int REGS_SOFTMAX = 216;
    static constexpr int REGS_OTHER = 72;
    static_assert(2 * 128 * REGS_SOFTMAX + 128 * REGS_OTHER <= NT * REGS_LAUNCH,
                  "setmaxnreg split must fit the launch's register file share");
    // K (or V) tile of stream u in stage s
    static constexpr int k_off(int s, int u) { return OFF_KV + s * STAGE_BYTES + u * KV_BYTES; }
    static constexpr int v_off(int s, int u) {
        return OFF_KV + s * STAGE_BYTES + (STREAMS + u) * KV_BYTES;
    }
    // penalty tile v (= h chunk * w chunks + w chunk) of stream u
    static constexpr int kxv_off(int u, int v) { return OFF_KXV + (u * MAXV + v) * KX_BYTES; }
};

struct TcParams {
    int Nq, Nkv;             // full attention: query / key tokens per (batch, head)
    float c_log2;            // scale * log2(e)
    void *o;                 // bf16 or f16, like the inputs
    unsigned *err;
    // neighborhood attention (grid T x Hg x W, row-major)
    int T, Hg, W;
    int kt, kh, kw;          // requested kernel
    int et, eh, ew;          // effective kernel
    int bt, bh, bw;          // query box
    int nbh, nbw2;           // boxes along h; box pairs along w
    int nbw;                 // boxes along w
    int KH;                  // key sub-box height (keys per tile = KH * 16)
    float penalty;           // bf16: power of two >= 2^100 with penalty * c_log2 >= 300
    // causal grouped-query prefill
    int Hq, Hkv, group;
    // full / causal: q, k, v are 4D tensor maps {D, N, heads, B}; o is written
    // through element strides (batch, head, row), D contiguous
    int H;                   // query heads (the batch of block row bh is bh / H)
    long long o_sb, o_sh, o_sn;
};

// Barrier block at OFF_BAR.
template <int NS>
struct Bars {
    uint64_t q_full;
    // K and V rings are released separately: a K stage as soon as the Q K^T
    // products that read it have completed, a V stage after its P V
    uint64_t k_full[NS], v_full[NS], k_empty[NS], v_empty[NS];
    uint64_t s_full[kNQ], s_free[kNQ], p_ready[kNQ], o_done[kNQ];
    uint64_t drain;
    uint32_t tmem_base;
    int abort;
};

// Per-query-tile geometry of the neighborhood path.
struct NaTile {
    int t0, h0, w0;          // box origin
    int u0t, u0h, u0w;       // union origin
    int ut, nhc, nwc;        // union t extent, h chunks, w chunks
    int ntiles;              // key tiles = ut * nhc * nwc (0 if the box is empty)
};

// a[t] for a per-query-tile array and a run-time t, by selects: indexing
// the array with a run-time value would place it in local memory
template <typename T>
__device__ __forceinline__ T pick(const T (&a)[kNQ], int t) {
    T r = a[0];
#pragma unroll
    for (int i = 1; i < kNQ; ++i)
        if (t == i) r = a[i];
    return r;
}

__device__ __forceinline__ NaTile na_tile(const TcParams &p, int pair, int t) {
    NaTile g;
    const int per_t = p.nbh * p.nbw2;
    const int bi_t = pair / per_t, bi_h = (pair / p.nbw2) % p.nbh, bi_w = (pair % p.nbw2) * 2 + t;
    g.t0 = bi_t * p.bt;
    g.h0 = bi_h * p.bh;
    g.w0 = bi_w * p.bw;
    if (bi_w >= p.nbw) {
        g.ntiles = 0;
        g.u0t = g.u0h = g.u0w = g.ut = g.nhc = g.nwc = 0;
        return g;
    }
    const int t1 = imin(g.t0 + p.bt, p.T) - 1, h1 = imin(g.h0 + p.bh, p.Hg) - 1,
              w1 = imin(g.w0 + p.bw, p.W) - 1;
    g.u0t = na_window_start(g.t0, p.T, p.kt);
    g.u0h = na_window_start(g.h0, p.Hg, p.kh);
    g.u0w = na_window_start(g.w0, p.W, p.kw);
    g.ut = na_window_start(t1, p.T, p.kt) + p.et - g.u0t;
    const int uh = na_window_start(h1, p.Hg, p.kh) + p.eh - g.u0h;
    const int uw = na_window_start(w1, p.W, p.kw) + p.ew - g.u0w;
    g.nhc = cdiv(uh, p.KH);
    g.nwc = cdiv(uw, kKW);
    g.ntiles = g.ut * g.nhc * g.nwc;
    return g;
}

// Key sub-box of tile j: origin (t, h, w).
__device__ __forceinline__ void na_key_box(const NaTile &g, int KH, int j, int &t, int &h, int &w) {
    const int wc = j % g.nwc;
    const int hc = (j / g.nwc) % g.nhc;
    const int tc = j / (g.nwc * g.nhc);
    t = g.u0t + tc;
    h = g.u0h + hc * KH;
    w = g.u0w + wc * kKW;
}

// KHC > 0 fixes the neighborhood key sub-box height (keys per tile = 16 KHC)
// at compile time, so the softmax's column loops and masks unroll without
// run-time tests; KHC = 0 takes it from the parameters.  F16: inputs, P and
// output in f16 instead of bf16 (same layouts; the MMA operand format flips).
template <int D, bool NA, bool CAUSAL, int KHC, bool F16>
__global__ void __launch_bounds__(TcCfg<D, NA>::NT, 1)
tc_attn_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
               const __grid_constant__ CUtensorMap tv, const TcParams p) {
    using C = TcCfg<D, NA>;
    static_assert(!(NA && CAUSAL), "causal prefill is a full-attention variant");
    static_assert(sizeof(Bars<C::NSTAGE>) <= 512, "barrier block must fit its reserved bytes");
    extern __shared__ uint8_t smem_raw[];
    // 1024-byte alignment for the 128-byte swizzle atoms
    uint8_t *smem = smem_raw + ((1024 - (ptx::smem_addr(smem_raw) & 1023)) & 1023);
    Bars<C::NSTAGE> *bars = reinterpret_cast<Bars<C::NSTAGE> *>(smem + C::OFF_BAR);
    volatile int *abort = &bars->abort;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int bh = blockIdx.y;
    // full attention: batch and head of this block row, and the K/V head (the
    // query head's KV head for grouped-query attention: contiguous groups of
    // Hq / Hkv query heads)
    const int fb = NA ? 0 : bh / p.H, fh = NA ? 0 : bh % p.H;
    const int fkh = CAUSAL ? fh / p.group : fh;

    // ---- per-CTA work description (identical in every role)
    int n_t[kNQ];
    int steps;
    NaTile g[kNQ];
    int q0 = 0;
    int BNt = kBN;                 // keys per tile
    if constexpr (NA) {
#pragma unroll
        for (int t = 0; t < kNQ; ++t) {
            g[t] = na_tile(p, blockIdx.x, t);
            n_t[t] = g[t].ntiles;
        }
        BNt = (KHC > 0 ? KHC : p.KH) * kKW;
        steps = imax(n_t[0], n_t[1]);
    } else if constexpr (CAUSAL) {
        // heaviest query blocks first; query tile t sees key tiles 0 .. its diagonal
        q0 = (gridDim.x - 1 - blockIdx.x) * (kNQ * kBM);
        const int all = cdiv(p.Nkv, kBN);
#pragma unroll
        for (int t = 0; t < kNQ; ++t)   // a query tile past the sequence's end has no work
            n_t[t] = q0 + t * kBM < p.Nq ? imin(all, (q0 + t * kBM) / kBN + 1) : 0;
        steps = imax(n_t[0], n_t[1]);
    } else {
        q0 = blockIdx.x * (kNQ * kBM);
        steps = cdiv(p.Nkv, kBN);
        n_t[0] = n_t[1] = steps;
    }

    if (threadIdx.x == 0) {
        ptx::mbar_init(&bars->q_full, 1);
        for (int s = 0; s < C::NSTAGE; ++s) {
            ptx::mbar_init(&bars->k_full[s], 1);
            ptx::mbar_init(&bars->v_full[s], 1);
            ptx::mbar_init(&bars->k_empty[s], 1);
            ptx::mbar_init(&bars->v_empty[s], 1);
        }
        for (int t = 0; t < kNQ; ++t) {
            ptx::mbar_init(&bars->s_full[t], 1);
            ptx::mbar_init(&bars->s_free[t], 128);
            ptx::mbar_init(&bars->p_ready[t], 128);
            ptx::mbar_init(&bars->o_done[t], 1);
        }
        ptx::mbar_init(&bars->drain, 1);
        bars->abort = 0;
        ptx::fence_barrier_init();
    }
    if constexpr (NA) {
        // query rows past the box (box smaller than 128 rows) hold zeros, not stale data
        const int rows = p.bt * p.bh * p.bw;
        if (rows < kBM) {
            for (int i = threadIdx.x; i < kNQ * C::PANELS * (kBM - rows) * 8; i += C::NT) {
                const int chunk = i % 8, r = rows + (i / 8) % (kBM - rows);
                const int pt = i / (8 * (kBM - rows));          // (tile, panel)
                *reinterpret_cast<uint4 *>(smem + C::OFF_Q + pt * C::PANEL_Q + r * 128 + chunk * 16) =
                    make_uint4(0, 0, 0, 0);
            }
        }
    }
    if constexpr (NA && !F16) {
        const int rows = p.bt * p.bh * p.bw;
        // one-hot window-offset channels of every query row: channel dh, then
        // bh + dw (rows past the box: all zero)
        for (int i = threadIdx.x; i < kNQ * kBM * 2; i += C::NT) {
            const int t = i / (kBM * 2), r = (i / 2) % kBM, half = i % 2;
            uint32_t w[4] = {0u, 0u, 0u, 0u};
            if (r < rows) {
                const int dh = (r / p.bw) % p.bh, dw = r % p.bw;
                const int ch[2] = {dh, p.bh + dw};
#pragma unroll
                for (int a = 0; a < 2; ++a) {
                    const int c = ch[a] - half * 8;
                    if (c >= 0 && c < 8) w[c >> 1] |= uint32_t(H16<F16>::kOne) << ((c & 1) * 16);
                }
            }
            *reinterpret_cast<uint4 *>(smem + C::OFF_QX + t * kBM * C::X_ROW + ptx::sw32_offset(r, half)) =
                make_uint4(w[0], w[1], w[2], w[3]);
        }
        // key-side penalty tiles: for key (h, w) of the sub-box of h chunk hc and
        // w chunk wc, channel dh holds -penalty if h lies outside the h window of
        // query offset dh, channel bh + dw likewise for w
        const typename H16<F16>::T negh = H16<F16>::from(-p.penalty);
        const uint32_t neg = uint32_t(*reinterpret_cast<const uint16_t *>(&negh));
#pragma unroll
        for (int u = 0; u < C::STREAMS; ++u) {
            if (n_t[u] == 0) continue;
            const int nv = g[u].nhc * g[u].nwc;
            for (int i = threadIdx.x; i < nv * BNt * 2; i += C::NT) {
                const int v = i / (BNt * 2), r = (i / 2) % BNt, half = i % 2;
                const int kh = g[u].u0h + (v / g[u].nwc) * (BNt / kKW) + r / kKW;
                const int kw = g[u].u0w + (v % g[u].nwc) * kKW + r % kKW;
                uint32_t w[4] = {0u, 0u, 0u, 0u};
#pragma unroll
                for (int cc = 0; cc < 8; ++cc) {
                    const int c = half * 8 + cc;
                    bool viol = false;
                    if (c < p.bh) {
                        const int sh = na_window_start(imin(g[u].h0 + c, p.Hg - 1), p.Hg, p.kh);
                        viol = unsigned(kh - sh) >= unsigned(p.eh);
                    } else if (c < p.bh + p.bw) {
                        const int sw = na_window_start(imin(g[u].w0 + c - p.bh, p.W - 1), p.W, p.kw);
                        viol = unsigned(kw - sw) >= unsigned(p.ew);
                    }
                    if (viol) w[cc >> 1] |= neg << ((cc & 1) * 16);
                }
                *reinterpret_cast<uint4 *>(smem + C::kxv_off(u, v) + ptx::sw32_offset(r, half)) =
                    make_uint4(w[0], w[1], w[2], w[3]);
            }
        }
        ptx::fence_proxy_async_smem();
    }
    if (warp == C::W_MMA) {
        ptx::tmem_alloc(&bars->tmem_base, C::TM_COLS);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = bars->tmem_base;

    if (warp >= C::NSOFT) {
        ptx::regs_decrease<C::REGS_OTHER>();
        if ((warp == C::W_LOAD || warp == C::W_LOADV) && lane == 0) {
            // ============================================= TMA loaders: one
            // thread streams Q and the K ring, another the V ring, so each
            // ring refills as soon as its own stage is released
            const int which = warp == C::W_LOAD ? 0 : 1;
            const CUtensorMap *tm = which == 0 ? &tk : &tv;
            uint64_t *full = which == 0 ? bars->k_full : bars->v_full;
            uint64_t *empty = which == 0 ? bars->k_empty : bars->v_empty;
            ptx::prefetch_tmap(tm);
            const uint64_t pol_kv = ptx::l2_policy_evict_last();
            if (which == 0) {
                ptx::prefetch_tmap(&tq);
                const uint64_t pol_q = ptx::l2_policy_evict_first();
                uint32_t qbytes = 0;
                if constexpr (NA) {
#pragma unroll
                    for (int t = 0; t < kNQ; ++t)
                        if (n_t[t] > 0) qbytes += C::PANELS * p.bt * p.bh * p.bw * 128;
                } else {
                    qbytes = kNQ * C::Q_BYTES;
                }
                ptx::mbar_arrive_expect_tx(&bars->q_full, qbytes);
#pragma unroll
                for (int t = 0; t < kNQ; ++t)
                    for (int pn = 0; pn < C::PANELS; ++pn) {
                        uint8_t *dst = smem + C::OFF_Q + t * C::Q_BYTES + pn * C::PANEL_Q;
                        if constexpr (NA) {
                            if (n_t[t] > 0)
                                ptx::tma_load_5d(dst, &tq, pn * 64, g[t].w0, g[t].h0, g[t].t0, bh,
                                                 &bars->q_full, pol_q);
                        } else {
                            ptx::tma_load_4d(dst, &tq, pn * 64, q0 + t * kBM, fh, fb, &bars->q_full,
                                             pol_q);
                        }
                    }
            }
            int issued = 0;
            for (int j = 0; j < steps; ++j) {
                const int s = j % C::NSTAGE;
                if (j >= C::NSTAGE &&
                    !ptx::mbar_wait_or_abort(&empty[s], ((j / C::NSTAGE) - 1) & 1, p.err, abort))
                    break;
                issued = j + 1;
                // a shared K/V stream (no neighborhood boxes) serves both query
                // tiles, so it runs for the longer of the two tile counts
                auto stream_has = [&](int u) { return NA ? j < n_t[u] : j < steps; };
                uint32_t bytes = 0;
#pragma unroll
                for (int u = 0; u < C::STREAMS; ++u)
                    if (stream_has(u)) bytes += C::PANELS * BNt * 128;
                ptx::mbar_arrive_expect_tx(&full[s], bytes);
#pragma unroll
                for (int u = 0; u < C::STREAMS; ++u) {
                    if (!stream_has(u)) continue;
                    for (int pn = 0; pn < C::PANELS; ++pn) {
                        uint8_t *dst =
                            smem + (which == 0 ? C::k_off(s, u) : C::v_off(s, u)) + pn * C::PANEL_KV;
                        if constexpr (NA) {
                            int kt_, kh_, kw_;
                            na_key_box(g[u], BNt / kKW, j, kt_, kh_, kw_);
                            ptx::tma_load_5d(dst, tm, pn * 64, kw_, kh_, kt_, bh, &full[s], pol_kv);
                        } else {
                            ptx::tma_load_4d(dst, tm, pn * 64, j * kBN, fkh, fb, &full[s], pol_kv);
                        }
                    }
                }
            }
            // after a timeout elsewhere: let the copies this thread issued land
            // (bounded) before the CTA's shared memory is released
            if (*abort) {
                if (which == 0) ptx::mbar_wait(&bars->q_full, 0, nullptr);
                for (int j = imax(0, issued - C::NSTAGE); j < issued; ++j)
                    ptx::mbar_wait(&full[j % C::NSTAGE], (j / C::NSTAGE) & 1, nullptr);
            }
        } else if (warp == C::W_MMA && lane == 0) {
            // ============================================= MMA issuer
            const uint32_t id_qk = ptx::idesc_16_f32(kBM, BNt, false, F16);
            const uint32_t id_pv = ptx::idesc_16_f32(kBM, D, true, F16);
            // Matrix descriptors are built once: a k-step, a stage or a tile only
            // moves the start-address field (bits 0-13, byte address >> 4, no
            // carry out of it below 256 KB), so each MMA costs one add here
            // instead of a rebuilt 64-bit descriptor on this single thread.
            constexpr uint32_t HI128 = ptx::desc_hi_sw128(1024), HI32 = ptx::desc_hi_sw32(256);
            const uint32_t dq0 = ptx::desc_lo_sw128(ptx::smem_addr(smem + C::OFF_Q), 16);
            const uint32_t dk0 = ptx::desc_lo_sw128(ptx::smem_addr(smem + C::k_off(0, 0)), 16);
            const uint32_t dv0 = ptx::desc_lo_sw128(ptx::smem_addr(smem + C::v_off(0, 0)), C::PANEL_KV);
            uint32_t dqx0 = 0, dkx0 = 0;
            int vq[kNQ], nv[kNQ];                // penalty tile of each tile's next Q K^T
#pragma unroll
            for (int t = 0; t < kNQ; ++t) {
                vq[t] = 0;
                nv[t] = 1;
            }
            if constexpr (NA) {
                dqx0 = ptx::desc_lo_sw32(ptx::smem_addr(smem + C::OFF_QX));
                dkx0 = ptx::desc_lo_sw32(ptx::smem_addr(smem + C::kxv_off(0, 0)));
#pragma unroll
                for (int t = 0; t < kNQ; ++t) nv[t] = imax(1, g[t].nhc * g[t].nwc);
            }
            const int nkv = BNt / 16;            // k-steps of P V
            auto issue_qk = [&](int t, int j) {
                const int s = j % C::NSTAGE;
                const uint32_t a0 = dq0 + uint32_t((t * C::Q_BYTES) >> 4);
                const uint32_t b0 =
                    dk0 + uint32_t((s * C::STAGE_BYTES + (C::STREAMS == 1 ? 0 : t) * C::KV_BYTES) >> 4);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t oa = ((kk >> 2) * C::PANEL_Q + (kk & 3) * 32) >> 4;
                    const uint32_t ob = ((kk >> 2) * C::PANEL_KV + (kk & 3) * 32) >> 4;
                    ptx::mma_ss(tmem + C::TM_S + t * kBN, ptx::desc_join(a0 + oa, HI128),
                                ptx::desc_join(b0 + ob, HI128), id_qk, kk > 0);
                }
                if constexpr (NA && !F16) {
                    // + window penalties: one more k-step over the 16 extra channels;
                    // QK_t(j) uses penalty tile j mod (h chunks x w chunks)
                    const uint32_t a = dqx0 + uint32_t((t * kBM * C::X_ROW) >> 4);
                    const uint32_t b = dkx0 + uint32_t(((t * C::MAXV + vq[t]) * C::KX_BYTES) >> 4);
                    if (++vq[t] == nv[t]) vq[t] = 0;
                    ptx::mma_ss(tmem + C::TM_S + t * kBN, ptx::desc_join(a, HI32), ptx::desc_join(b, HI32),
                                id_qk, 1u);
                }
                ptx::tc_commit(&bars->s_full[t]);
            };
            auto issue_pv = [&](int t, int j) {
                const int s = j % C::NSTAGE;
                const uint32_t b0 =
                    dv0 + uint32_t((s * C::STAGE_BYTES + (C::STREAMS == 1 ? 0 : t) * C::KV_BYTES) >> 4);
                const uint32_t a0 = tmem + C::TM_P + t * C::PSTRIDE;
#pragma unroll
                for (int kk = 0; kk < kBN / 16; ++kk) {
                    if (kk >= nkv) break;
                    ptx::mma_ts(tmem + C::TM_O + t * D, a0 + kk * 8,
                                ptx::desc_join(b0 + uint32_t(kk * (2048 >> 4)), HI128), id_pv,
                                (j > 0 || kk > 0) ? 1u : 0u);
                }
                ptx::tc_commit(&bars->o_done[t]);
            };
            bool ok = ptx::mbar_wait_or_abort(&bars->q_full, 0, p.err, abort) &&
                      (steps == 0 || ptx::mbar_wait_or_abort(&bars->k_full[0], 0, p.err, abort));
            ptx::tc_fence_after();
            if (ok) {
#pragma unroll
                for (int t = 0; t < kNQ; ++t)
                    if (n_t[t] > 0) issue_qk(t, 0);
                if (steps > 0) ptx::tc_commit(&bars->k_empty[0]);
            }
            for (int j = 0; ok && j < steps; ++j) {
                const int s = j % C::NSTAGE;
                const uint32_t ph = (j / C::NSTAGE) & 1;
                const int s1 = (j + 1) % C::NSTAGE;
                const uint32_t ph1 = ((j + 1) / C::NSTAGE) & 1;
                bool v_ready = false, k1_ready = false;
                auto wait_k1 = [&]() {
                    if (!k1_ready) {
                        ok = ok && ptx::mbar_wait_or_abort(&bars->k_full[s1], ph1, p.err, abort);
                        k1_ready = true;
                    }
                };
                auto wait_v = [&]() {
                    if (!v_ready) {
                        ok = ok && ptx::mbar_wait_or_abort(&bars->v_full[s], ph, p.err, abort);
                        v_ready = true;
                    }
                };
                if constexpr (C::SEP_P) {
                    // next S as soon as the softmax holds the current one in registers
#pragma unroll
                    for (int t = 0; t < kNQ; ++t) {
                        if (!ok) break;
                        if (j + 1 >= n_t[t]) continue;
                        ok = ptx::mbar_wait_or_abort(&bars->s_free[t], j & 1, p.err, abort);
                        wait_k1();
                        if (!ok) break;
                        ptx::tc_fence_after();
                        issue_qk(t, j + 1);
                    }
#pragma unroll
                    for (int t = 0; t < kNQ; ++t) {
                        if (!ok) break;
                        if (j >= n_t[t]) continue;
                        ok = ptx::mbar_wait_or_abort(&bars->p_ready[t], j & 1, p.err, abort);
                        wait_v();
                        if (!ok) break;
                        ptx::tc_fence_after();
                        issue_pv(t, j);
                    }
                } else {
#pragma unroll
                    for (int t = 0; t < kNQ; ++t) {
                        if (!ok) break;
                        if (j >= n_t[t]) continue;
                        ok = ptx::mbar_wait_or_abort(&bars->p_ready[t], j & 1, p.err, abort);
                        wait_v();
                        if (!ok) break;
                        ptx::tc_fence_after();
                        issue_pv(t, j);
                        if (j + 1 < n_t[t]) {
                            wait_k1();
                            if (!ok) break;
                            ptx::tc_fence_after();
                            issue_qk(t, j + 1);
                        }
                    }
                }
                // every Q K^T of step j + 1 and every P V of step j is issued
                if (j + 1 < steps) ptx::tc_commit(&bars->k_empty[s1]);
                ptx::tc_commit(&bars->v_empty[s]);
            }
            // drain: every MMA this thread issued has completed before TMEM is freed
            ptx::tc_commit(&bars->drain);
            ptx::mbar_wait(&bars->drain, 0, p.err);
        }
    } else {
        // ================================================= softmax warpgroups
        ptx::regs_increase<C::REGS_SOFTMAX>();
        const int t = warp >> 2;                 // query tile
        const int quarter = warp & 3;            // TMEM lanes [32 quarter, 32 quarter + 32)
        const int row = quarter * 32 + lane;     // query row within the tile
        const uint32_t lane_base = tmem + (uint32_t(quarter * 32) << 16);
        const uint32_t s_addr = lane_base + C::TM_S + t * kBN;
        const uint32_t p_addr = lane_base + C::TM_P + t * C::PSTRIDE;
        const uint32_t o_addr = lane_base + C::TM_O + t * D;
        const float cl = p.c_log2;

        // query of this row (neighborhood path) and its window
        int qt = 0, qh = 0, qw = 0, wst = 0, wsh = 0, wsw = 0;
        bool qvalid;
        const NaTile gt = pick(g, t);           // this warp's tile, in registers
        const int nt = pick(n_t, t);
        if constexpr (NA) {
            const int dt = row / (p.bh * p.bw), dh = (row / p.bw) % p.bh, dw = row % p.bw;
            qt = gt.t0 + dt;
            qh = gt.h0 + dh;
            qw = gt.w0 + dw;
            qvalid = nt > 0 && row < p.bt * p.bh * p.bw && qt < p.T && qh < p.Hg && qw < p.W;
            wst = na_window_start(imin(qt, p.T - 1), p.T, p.kt);
            if constexpr (F16) {
                wsh = na_window_start(imin(qh, p.Hg - 1), p.Hg, p.kh);
                wsw = na_window_start(imin(qw, p.W - 1), p.W, p.kw);
            }
        } else {
            qvalid = q0 + t * kBM + row < p.Nq;
        }

        float m = -INFINITY, l = 0.f;
        bool ok = true;
        // neighborhood: key sub-box counters (w fastest, then h, then t)
        int tc = 0, hc = 0, wc = 0;
        for (int j = 0; j < nt; ++j) {
            if (!__all_sync(0xffffffffu,
                            ptx::mbar_wait_or_abort(&bars->s_full[t], j & 1, p.err, abort))) {
                ok = false;
                break;
            }
            ptx::tc_fence_after();

            // ---- neighborhood: the h and w window penalties are already in S
            //      (extra MMA channels); a row whose t window misses this key
            //      sub-box's frame gets P = 0 below.  (Skipping sub-boxes that
            //      none of a warp's 32 windows reaches measured slower than
            //      computing them: the MMAs run anyway and the test costs issue
            //      slots on the critical path.)
            bool t_ok = true;
            int kh0 = 0, kw0 = 0;                // key sub-box origin along h and w
            if constexpr (NA) {
                const int kt_ = gt.u0t + tc;
                kh0 = gt.u0h + hc * (BNt / kKW);
                kw0 = gt.u0w + wc * kKW;
                if (++wc == gt.nwc) {
                    wc = 0;
                    if (++hc == gt.nhc) {
                        hc = 0;
                        ++tc;
                    }
                }
                t_ok = qvalid && unsigned(kt_ - wst) < unsigned(p.et);
            }

            float sv[kBN];
#pragma unroll
            for (int c = 0; c < kBN / 32; ++c)
                if (c * 32 < BNt)
                    ptx::tmem_ld32(s_addr + c * 32, *reinterpret_cast<uint32_t(*)[32]>(&sv[c * 32]));
            ptx::tmem_wait_ld();
            if constexpr (C::SEP_P) {
                // S_t is in registers: the next QK_t may overwrite it
                ptx::tc_fence_before();
                ptx::mbar_arrive(&bars->s_free[t]);
            }

            // ---- mask: keys that do not exist in this tile
            if constexpr (NA) {
                // columns past this tile's keys (N = KH * 16 < 128) hold stale
                // values: whole 16-column groups, warp-uniform
#pragma unroll
                for (int gq = 0; gq < kBN / 16; ++gq)
                    if (gq * 16 >= BNt) {
#pragma unroll
                        for (int i = 0; i < 16; ++i) sv[gq * 16 + i] = -INFINITY;
                    }
                if constexpr (F16) {
                    // f16: the h and w window tests per key.  Key e of the
                    // (1, KH, 16) sub-box sits at h = kh0 + e / 16, w = kw0 + e % 16;
                    // wm / hm hold the in-window w columns / h rows of this row.
                    const int lw = wsw - kw0, lh = wsh - kh0;
                    const int aw = imax(lw, 0), bw = imin(lw + p.ew, kKW);
                    const int ah = imax(lh, 0), bh_ = imin(lh + p.eh, kBN / kKW);
                    const uint32_t wm = aw < bw ? ((1u << bw) - 1u) & ~((1u << aw) - 1u) : 0u;
                    const uint32_t hm = ah < bh_ ? ((1u << bh_) - 1u) & ~((1u << ah) - 1u) : 0u;
#pragma unroll
                    for (int gq = 0; gq < kBN / 16; ++gq) {
                        const bool hin = (hm >> gq) & 1u;
#pragma unroll
                        for (int i = 0; i < 16; ++i)
                            if (!hin || !((wm >> i) & 1u)) sv[gq * 16 + i] = -INFINITY;
                    }
                }
            } else {
                int valid = p.Nkv - j * kBN;           // keys of this tile inside the sequence
                if constexpr (CAUSAL) {
                    // the last tile is the diagonal one (query tile and key tile
                    // start at the same position): key e is visible to row `row`
                    // iff e <= row
                    if (j == nt - 1) {
#pragma unroll
                        for (int e = 0; e < kBN; ++e)
                            if (e > row || e >= valid) sv[e] = -INFINITY;
                        valid = kBN;
                    }
                }
                if (valid < kBN) {
#pragma unroll
                    for (int e = 0; e < kBN; ++e)
                        if (e >= valid) sv[e] = -INFINITY;
                }
            }

            // P = 2^(x - m) in 16-bit into TMEM; returns the tile's row sum (fp32)
            auto emit_p = [&](float nmu) -> float {
                float acc[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) acc[i] = 0.f;
#pragma unroll
                for (int c = 0; c < kBN / 32; ++c) {
                    if (c * 32 >= BNt) break;
                    uint32_t pk[16];
                    // the upper 16 keys of the last 32-key chunk may lie past the tile
                    const int ne = (c * 32 + 32 <= BNt) ? 16 : 8;
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        if (e >= 8 && ne == 8) {
                            pk[e] = 0u;
                            continue;
                        }
                        float x0, x1;
                        ptx::ffma2(x0, x1, sv[c * 32 + 2 * e], sv[c * 32 + 2 * e + 1], cl, cl, nmu,
                                   nmu);
                        const float p0 = ptx::ex2(x0), p1 = ptx::ex2(x1);
                        ptx::fadd2(acc[(2 * e) & 7], acc[(2 * e + 1) & 7], acc[(2 * e) & 7],
                                   acc[(2 * e + 1) & 7], p0, p1);
                        pk[e] = H16<F16>::pack(p0, p1);
                    }
                    ptx::tmem_st16(p_addr + c * 16, pk);
                }
                return ((acc[0] + acc[1]) + (acc[2] + acc[3])) + ((acc[4] + acc[5]) + (acc[6] + acc[7]));
            };

            // ---- fast path: exponentiate against the running maximum m as it
            //      stands, with no tile maximum.  P only has to stay finite in its
            //      16-bit type, not below 1: a tile whose row sum exceeds 2^24 (2^15
            //      for f16, whose largest finite value is 65504) or is not finite
            //      (scores far above m, or m still the garbage of a row whose
            //      first tiles were all outside its window) is redone below
            //      against its own maximum.  After the first tiles m is close to
            //      the row maximum and the redo almost never runs.
            bool fast = j > 0 && __all_sync(0xffffffffu, !(t_ok && m == -INFINITY));
            bool waited = false;                 // o_done of step j - 1 observed
            if (fast) {
                if constexpr (C::SEP_P) {
                    // P_t has columns of its own: the previous P V must have read them
                    if (!__all_sync(0xffffffffu, ptx::mbar_wait_or_abort(&bars->o_done[t], (j - 1) & 1,
                                                                         p.err, abort))) {
                        ok = false;
                        break;
                    }
                    ptx::tc_fence_after();
                    waited = true;
                }
                const float lt = emit_p(t_ok ? -m : -INFINITY);
                if (__any_sync(0xffffffffu, !(lt <= (F16 ? 32768.f : 16777216.f))))
                    fast = false;                 // redo the tile (P is rewritten below)
                else
                    l += lt;
            }

            if (!fast) {
                // ---- tile maximum
                float mx[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) mx[i] = fmaxf(sv[i], sv[8 + i]);
#pragma unroll
                for (int e = 16; e < kBN; e += 16)
#pragma unroll
                    for (int i = 0; i < 8; ++i) mx[i] = ptx::fmax3(mx[i], sv[e + i], sv[e + 8 + i]);
                const float tmax = ptx::fmax3(ptx::fmax3(mx[0], mx[1], mx[2]),
                                              ptx::fmax3(mx[3], mx[4], mx[5]), fmaxf(mx[6], mx[7]));
                const float mt = t_ok ? tmax * cl : -INFINITY;   // cl > 0: max commutes with the scaling

                // ---- the previous P V must be done before O is rescaled or P_t rewritten
                const bool want = j == 0 || mt > m + 8.f;   // this row moves its maximum
                const bool any_want = __any_sync(0xffffffffu, want);
                if (j > 0 && !waited && (C::SEP_P || any_want)) {
                    if (!__all_sync(0xffffffffu, ptx::mbar_wait_or_abort(&bars->o_done[t], (j - 1) & 1,
                                                                         p.err, abort))) {
                        ok = false;
                        break;
                    }
                    ptx::tc_fence_after();
                }
                // ---- running maximum (moved lazily) and O rescale in TMEM
                if (j == 0) {
                    m = mt;
                } else if (any_want) {
                    // rows that move m scale their O row; the others multiply by 1
                    const float f = want ? ptx::ex2(m - mt) : 1.f;   // m == -inf -> 0
#pragma unroll
                    for (int c = 0; c < D / 32; ++c) {
                        uint32_t ov[32];
                        ptx::tmem_ld32(o_addr + c * 32, ov);
                        ptx::tmem_wait_ld();
#pragma unroll
                        for (int e = 0; e < 32; e += 2) {
                            float a0, a1;
                            ptx::ffma2(a0, a1, __uint_as_float(ov[e]), __uint_as_float(ov[e + 1]), f,
                                       f, 0.f, 0.f);
                            ov[e] = __float_as_uint(a0);
                            ov[e + 1] = __float_as_uint(a1);
                        }
                        ptx::tmem_st32(o_addr + c * 32, ov);
                    }
                    if (want) {
                        l *= f;
                        m = mt;
                    }
                }
                // (a row whose t window misses this key sub-box gets P = 0)
                l += emit_p(!t_ok ? -INFINITY : (m == -INFINITY) ? 0.f : -m);
            }
            ptx::tmem_wait_st();
            ptx::tc_fence_before();
            ptx::mbar_arrive(&bars->p_ready[t]);
        }

        // ---- epilogue: O / l -> bf16 -> global
        if (ok && nt > 0 &&
            __all_sync(0xffffffffu,
                       ptx::mbar_wait_or_abort(&bars->o_done[t], (nt - 1) & 1, p.err, abort))) {
            ptx::tc_fence_after();
            const float inv = 1.f / l;
            typename H16<F16>::T *orow = nullptr;
            if (qvalid) {
                size_t idx;
                if constexpr (NA)
                    idx = ((size_t(bh) * (size_t(p.T) * p.Hg * p.W)) + (size_t(qt) * p.Hg + qh) * p.W + qw) * D;
                else
                    idx = size_t(fb * p.o_sb + fh * p.o_sh + (long long)(q0 + t * kBM + row) * p.o_sn);
                orow = static_cast<typename H16<F16>::T *>(p.o) + idx;
            }
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
                uint32_t ov[32];
                ptx::tmem_ld32(o_addr + c * 32, ov);
                ptx::tmem_wait_ld();
                if (qvalid) {
                    uint4 w4[4];
                    uint32_t *wp = reinterpret_cast<uint32_t *>(w4);
#pragma unroll
                    for (int e = 0; e < 16; ++e)
                        wp[e] = H16<F16>::pack(__uint_as_float(ov[2 * e]) * inv,
                                            __uint_as_float(ov[2 * e + 1]) * inv);
                    uint4 *dst = reinterpret_cast<uint4 *>(orow + c * 32);
#pragma unroll
                    for (int e = 0; e < 4; ++e) dst[e] = w4[e];
                }
            }
        }
    }

    // ---- teardown: all TMEM traffic done before the owner warp frees it
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == C::W_MMA) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, C::TM_COLS);
    }
}

// ---------------------------------------------------- single-tile self test
//
// One CTA: S = Q K^T + Q[:, :16] K[:, :16]^T (the first term from 128-byte
// swizzled K-major operands, the second from 32-byte swizzled copies -- the
// layout of the neighborhood kernel's window-penalty channels) and O = P V
// (P from TMEM, V MN-major in shared memory) for one 128 x 128 tile, written
// out in fp32: the MMA forms of the attention kernels in isolation.
template <int D>
__global__ void __launch_bounds__(160, 1)
tc_selftest_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                   const __grid_constant__ CUtensorMap tv, const __nv_bfloat16 *qg,
                   const __nv_bfloat16 *kg, const __nv_bfloat16 *P, float *S_out, float *O_out,
                   unsigned *err) {
    constexpr int PANELS = D / 64;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024 - (ptx::smem_addr(smem_raw) & 1023)) & 1023);
    uint8_t *sq = smem, *sk = smem + PANELS * 16384, *svv = smem + 2 * PANELS * 16384;
    // 32-byte-swizzled copies of the first 16 channels of q and k (the layout of
    // the extra window-penalty operands of the neighborhood kernel)
    uint8_t *sqx = smem + 3 * PANELS * 16384, *skx = sqx + 4096;
    for (int i = threadIdx.x; i < 2 * 128 * 2; i += blockDim.x) {
        const int which = i / 256, r = (i / 2) % 128, half = i % 2;
        const __nv_bfloat16 *src = (which == 0 ? qg : kg) + r * D + half * 8;
        *reinterpret_cast<uint4 *>((which == 0 ? sqx : skx) + ptx::sw32_offset(r, half)) =
            *reinterpret_cast<const uint4 *>(src);
    }
    ptx::fence_proxy_async_smem();
    __shared__ uint64_t bar_load, bar_mma, bar_p;
    __shared__ uint32_t tmem_base;
    __shared__ int abort;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        ptx::mbar_init(&bar_load, 1);
        ptx::mbar_init(&bar_mma, 1);
        ptx::mbar_init(&bar_p, 128);
        abort = 0;
        ptx::fence_barrier_init();
    }
    if (warp == 4) {
        ptx::tmem_alloc(&tmem_base, 512);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = tmem_base;   // S at col 0, O at col 256
    if (warp == 4) {
        if (lane == 0) {
            ptx::mbar_arrive_expect_tx(&bar_load, 3 * PANELS * 16384);
            for (int pn = 0; pn < PANELS; ++pn) {
                ptx::tma_load_3d(sq + pn * 16384, &tq, pn * 64, 0, 0, &bar_load, 0);
                ptx::tma_load_3d(sk + pn * 16384, &tk, pn * 64, 0, 0, &bar_load, 0);
                ptx::tma_load_3d(svv + pn * 16384, &tv, pn * 64, 0, 0, &bar_load, 0);
            }
            bool ok = ptx::mbar_wait_or_abort(&bar_load, 0, err, &abort);
            ptx::tc_fence_after();
            if (ok) {
                const uint32_t id_qk = ptx::idesc_bf16_f32(128, 128, false);
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t off = (kk & 3) * 32;
                    const uint64_t a = ptx::smem_desc_sw128(ptx::smem_addr(sq) + (kk >> 2) * 16384 + off, 16, 1024);
                    const uint64_t b = ptx::smem_desc_sw128(ptx::smem_addr(sk) + (kk >> 2) * 16384 + off, 16, 1024);
                    ptx::mma_ss(tmem, a, b, id_qk, kk > 0);
                }
                ptx::mma_ss(tmem, ptx::smem_desc_sw32(ptx::smem_addr(sqx), 256),
                            ptx::smem_desc_sw32(ptx::smem_addr(skx), 256), id_qk, 1);
                ptx::tc_commit(&bar_mma);
                ok = ptx::mbar_wait_or_abort(&bar_p, 0, err, &abort);
                ptx::tc_fence_after();
                if (ok) {
                    const uint32_t id_pv = ptx::idesc_bf16_f32(128, D, true);
                    for (int kk = 0; kk < 8; ++kk) {
                        const uint64_t b = ptx::smem_desc_sw128(ptx::smem_addr(svv) + kk * 2048, 16384, 1024);
                        ptx::mma_ts(tmem + 256, tmem + 128 + kk * 8, b, id_pv, kk > 0);
                    }
                }
                ptx::tc_commit(&bar_mma);
            }
        }
    } else {
        // 128 threads: write P (bf16) into TMEM columns [128, 192) after S is done,
        // then read S and O back.
        const int row = warp * 32 + lane;
        const uint32_t lb = tmem + (uint32_t(warp * 32) << 16);
        bool ok = __all_sync(0xffffffffu, ptx::mbar_wait_or_abort(&bar_mma, 0, err, &abort));
        ptx::tc_fence_after();
        if (ok) {
            for (int c = 0; c < 4; ++c) {
                uint32_t sv[32];
                ptx::tmem_ld32(lb + c * 32, sv);
                ptx::tmem_wait_ld();
                for (int e = 0; e < 32; ++e) S_out[row * 128 + c * 32 + e] = __uint_as_float(sv[e]);
            }
            for (int c = 0; c < 4; ++c) {
                uint32_t pk[16];
                const uint32_t *src = reinterpret_cast<const uint32_t *>(P + row * 128 + c * 32);
                for (int e = 0; e < 16; ++e) pk[e] = src[e];
                ptx::tmem_st16(lb + 128 + c * 16, pk);
            }
            ptx::tmem_wait_st();
        }
        ptx::tc_fence_before();
        ptx::mbar_arrive(&bar_p);
        if (ok) ok = __all_sync(0xffffffffu, ptx::mbar_wait_or_abort(&bar_mma, 1, err, &abort));
        ptx::tc_fence_after();
        if (ok) {
            for (int c = 0; c < D / 32; ++c) {
                uint32_t ov[32];
                ptx::tmem_ld32(lb + 256 + c * 32, ov);
                ptx::tmem_wait_ld();
                for (int e = 0; e < 32; ++e) O_out[row * D + c * 32 + e] = __uint_as_float(ov[e]);
            }
        }
    }
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 4) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, 512);
    }
}

// ------------------------------------------------------------- host side

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
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

// 16-bit (bf16 or f16) tensor map with 128-byte swizzle; dims/box innermost
// first (dims[0] = D).
bool make_tmap(CUtensorMap *m, const void *base, int rank, const uint64_t *dims,
               const uint32_t *box, bool f16 = false) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t gdim[5], gstride[4];
    cuuint32_t bdim[5], estr[5];
    uint64_t stride = 2;
    for (int i = 0; i < rank; ++i) {
        gdim[i] = dims[i];
        bdim[i] = box[i];
        estr[i] = 1;
        if (i > 0) gstride[i - 1] = stride;
        stride *= dims[i];
    }
    return fn(m, f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank,
              const_cast<void *>(base), gdim, gstride,
              bdim, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int D, bool NA, bool CAUSAL = false, int KHC = 0, bool F16 = false>
attn_status_t launch_tc(const Ctx &c, const CUtensorMap &tq, const CUtensorMap &tk,
                        const CUtensorMap &tv, const TcParams &p, dim3 grid) {
    using C = TcCfg<D, NA>;
    static int done_mask = 0;
    static int regs = -1;
    auto kern = tc_attn_kernel<D, NA, CAUSAL, KHC, F16>;
    if (!ensure_smem_attr(reinterpret_cast<const void *>(kern), C::SMEM, c.device, &done_mask))
        return ATTN_ERR_RESOURCE;
    // The warpgroups re-split the launch's register file with setmaxnreg; the
    // split is only valid for the per-thread count it was computed for.
    if (regs < 0) {
        cudaFuncAttributes fa;
        if (cudaFuncGetAttributes(&fa, reinterpret_cast<const void *>(kern)) != cudaSuccess) {
            cudaGetLastError();
            return ATTN_ERR_CUDA;
        }
        regs = fa.numRegs;
    }
    if (regs != C::REGS_LAUNCH) return ATTN_ERR_UNSUPPORTED;
    kern<<<grid, C::NT, C::SMEM, c.stream>>>(tq, tk, tv, p);
    return launch_status(NA ? kFamTcNa : kFamTcFlash);
}

// Query box and key sub-box height for the neighborhood path: at most 128
// queries per box, minimising the (query row, key) slots the MMAs compute over
// all boxes (boxes x tiles x (KH*16 + per-tile overhead)).
bool plan_na(int T, int Hg, int W, const int kern[3], int &bt, int &bh, int &bw, int &KH) {
    const int ext[3] = {T, Hg, W};
    double best = -1;
    for (int cbt = 1; cbt <= imin(T, 128); ++cbt)
        for (int cbh = 1; cbh <= imin(Hg, 128 / cbt); ++cbh)
            for (int cbw = 1; cbw <= imin(W, 128 / (cbt * cbh)); ++cbw) {
                if (cbt * cbh * cbw < imin(64, T * Hg * W)) continue;   // keep MMA rows busy
                if (cbh + cbw > 16) continue;                // h and w offsets fit 16 channels
                // key tiles of 64..128 keys keep the MMAs large enough to amortise
                // the per-tile barrier round trips
                for (int ckh = imin(4, imin(kern[1], Hg) + cbh - 1); ckh <= 8; ++ckh) {
                    // distinct key penalty tiles of a box (h chunks x w chunks) must fit
                    const int nh_max = cdiv(imin(cbh + imin(kern[1], Hg) - 1, Hg), ckh);
                    const int nw_max = cdiv(imin(cbw + imin(kern[2], W) - 1, W), kKW);
                    if (nh_max * nw_max > 6) continue;
                    // total key slots over all boxes = sum_t(ut) * sum_h(nhc) * sum_w(nwc) * KH*16
                    const int b[3] = {cbt, cbh, cbw};
                    double axis[3];
                    for (int a = 0; a < 3; ++a) {
                        const int keff = imin(kern[a], ext[a]);
                        double acc = 0;
                        for (int i0 = 0; i0 < ext[a]; i0 += b[a]) {
                            const int i1 = imin(i0 + b[a], ext[a]) - 1;
                            const int u = na_window_start(i1, ext[a], kern[a]) + keff -
                                          na_window_start(i0, ext[a], kern[a]);
                            acc += a == 0 ? u : a == 1 ? cdiv(u, ckh) : cdiv(u, kKW);
                        }
                        axis[a] = acc;
                    }
                    const int nbw = cdiv(W, cbw);
                    // odd box count along w leaves one query tile idle per (t, h) box row
                    const double w_pairs_waste = (nbw & 1) ? double(nbw + 1) / nbw : 1.0;
                    // every box is one 128-row query tile: computed (row, key) slots
                    // (a tile costs its key slots plus a fixed overhead of ~32 key slots)
                    const double cost = axis[0] * axis[1] * axis[2] * (ckh * kKW + 32) * w_pairs_waste;
                    if (best < 0 || cost < best) {
                        best = cost;
                        bt = cbt; bh = cbh; bw = cbw; KH = ckh;
                    }
                }
            }
    return best > 0;
}

// Plans are cached per (grid, kernel): the search is a few thousand candidates.
struct NaPlan {
    int bt, bh, bw, KH;
    bool ok;
};

NaPlan cached_plan(int T, int Hg, int W, const int kern[3]) {
    struct Entry {
        int key[6];
        NaPlan plan;
    };
    static std::mutex mu;
    static Entry cache[64];
    static int used = 0;
    const int key[6] = {T, Hg, W, kern[0], kern[1], kern[2]};
    std::lock_guard<std::mutex> lock(mu);
    for (int i = 0; i < used; ++i) {
        bool same = true;
        for (int a = 0; a < 6; ++a) same = same && cache[i].key[a] == key[a];
        if (same) return cache[i].plan;
    }
    NaPlan pl{};
    pl.ok = plan_na(T, Hg, W, kern, pl.bt, pl.bh, pl.bw, pl.KH);
    Entry &e = cache[used < 64 ? used++ : 63];
    for (int a = 0; a < 6; ++a) e.key[a] = key[a];
    e.plan = pl;
    return pl;
}

}  // namespace

// 4D map {D, N, heads, B} over a tensor with element strides (row, head,
// batch) and D contiguous; 128-byte swizzle, box {64, 128, 1, 1}.
bool make_tmap4(CUtensorMap *m, const void *base, int D, int N, int heads, int B,
                const TensorStrides &st, bool f16) {
    auto fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t gdim[4] = {cuuint64_t(D), cuuint64_t(N), cuuint64_t(heads), cuuint64_t(B)};
    const cuuint64_t gstride[3] = {cuuint64_t(st.n) * 2, cuuint64_t(st.h) * 2, cuuint64_t(st.b) * 2};
    const cuuint32_t box[4] = {64, kBM, 1, 1};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    return fn(m, f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4,
              const_cast<void *>(base), gdim, gstride, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool tc_full_supported(int B, int H, int Nq, int Nkv, int D) {
    return (D == 64 || D == 128) && B * H <= 65535 && Nq >= 1 && Nkv >= 1 && encode_fn() != nullptr;
}

attn_status_t tc_full(const Ctx &c, attn_dtype_t dt, const void *q, const void *k, const void *v,
                      void *o, int B, int H, int Nq, int Nkv, int D, float scale,
                      const TensorStrides *st) {
    const bool f16 = dt == ATTN_F16;
    TensorStrides s4[4];                 // q, k, v, o
    for (int i = 0; i < 4; ++i) {
        const int n = i == 0 || i == 3 ? Nq : Nkv;
        s4[i] = st ? st[i] : TensorStrides{(long long)H * n * D, (long long)n * D, D};
    }
    CUtensorMap tq, tk, tv;
    // a layout the tensor-map encoder refuses goes to the strided SIMT kernel
    if (!make_tmap4(&tq, q, D, Nq, H, B, s4[0], f16) || !make_tmap4(&tk, k, D, Nkv, H, B, s4[1], f16) ||
        !make_tmap4(&tv, v, D, Nkv, H, B, s4[2], f16))
        return ATTN_ERR_UNSUPPORTED;
    TcParams p{};
    p.Nq = Nq;
    p.Nkv = Nkv;
    p.c_log2 = scale * kLog2e;
    p.o = o;
    p.err = c.err;
    p.H = H;
    p.o_sb = s4[3].b; p.o_sh = s4[3].h; p.o_sn = s4[3].n;
    const dim3 grid(cdiv(Nq, kNQ * kBM), B * H);
    if (f16)
        return D == 128 ? launch_tc<128, false, false, 0, true>(c, tq, tk, tv, p, grid)
                        : launch_tc<64, false, false, 0, true>(c, tq, tk, tv, p, grid);
    return D == 128 ? launch_tc<128, false>(c, tq, tk, tv, p, grid)
                    : launch_tc<64, false>(c, tq, tk, tv, p, grid);
}

attn_status_t tc_causal_gqa(const Ctx &c, attn_dtype_t dt, const void *q, const void *k,
                            const void *v, void *o, int B, int Hq, int Hkv, int N, int D,
                            float scale, const TensorStrides *st) {
    const bool f16 = dt == ATTN_F16;
    CUtensorMap tq, tk, tv;
    const TensorStrides dq{(long long)Hq * N * D, (long long)N * D, D};
    const TensorStrides dkv{(long long)Hkv * N * D, (long long)N * D, D};
    const TensorStrides sq = st ? st[0] : dq, sk = st ? st[1] : dkv, sv = st ? st[2] : dkv,
                        so = st ? st[3] : dq;
    // a layout the tensor-map encoder refuses goes to the strided SIMT kernel
    if (!make_tmap4(&tq, q, D, N, Hq, B, sq, f16) || !make_tmap4(&tk, k, D, N, Hkv, B, sk, f16) ||
        !make_tmap4(&tv, v, D, N, Hkv, B, sv, f16))
        return ATTN_ERR_UNSUPPORTED;
    TcParams p{};
    p.Nq = N;
    p.Nkv = N;
    p.c_log2 = scale * kLog2e;
    p.o = o;
    p.err = c.err;
    p.Hq = Hq;
    p.Hkv = Hkv;
    p.group = Hq / Hkv;
    p.H = Hq;
    p.o_sb = so.b; p.o_sh = so.h; p.o_sn = so.n;
    const dim3 grid(cdiv(N, kNQ * kBM), B * Hq);
    if (f16)
        return D == 128 ? launch_tc<128, false, true, 0, true>(c, tq, tk, tv, p, grid)
                        : launch_tc<64, false, true, 0, true>(c, tq, tk, tv, p, grid);
    return D == 128 ? launch_tc<128, false, true>(c, tq, tk, tv, p, grid)
                    : launch_tc<64, false, true>(c, tq, tk, tv, p, grid);
}

bool tc_na3d_supported(int B, int H, int T, int Hg, int W, int D, const int kernel[3]) {
    return D == 64 && B * H <= 65535 && encode_fn() != nullptr &&
           cached_plan(T, Hg, W, kernel).ok;
}

attn_status_t tc_na3d(const Ctx &c, attn_dtype_t dt, const void *q, const void *k, const void *v,
                      void *o, int B, int H, int T, int Hg, int W, int D, const int kernel[3],
                      float scale) {
    const bool f16 = dt == ATTN_F16;
    TcParams p{};
    const NaPlan pl = cached_plan(T, Hg, W, kernel);
    if (!pl.ok) return ATTN_ERR_UNSUPPORTED;
    p.bt = pl.bt; p.bh = pl.bh; p.bw = pl.bw; p.KH = pl.KH;
    CUtensorMap tq, tk, tv;
    const uint64_t dims[5] = {uint64_t(D), uint64_t(W), uint64_t(Hg), uint64_t(T), uint64_t(B) * H};
    const uint32_t qbox[5] = {64, uint32_t(p.bw), uint32_t(p.bh), uint32_t(p.bt), 1};
    const uint32_t kbox[5] = {64, uint32_t(kKW), uint32_t(p.KH), 1, 1};
    if (!make_tmap(&tq, q, 5, dims, qbox, f16) || !make_tmap(&tk, k, 5, dims, kbox, f16) ||
        !make_tmap(&tv, v, 5, dims, kbox, f16))
        return ATTN_ERR_CUDA;
    p.c_log2 = scale * kLog2e;
    // bf16 penalty per violated axis: a power of two (exact in bf16), at least
    // 2^100 and with penalty * scale * log2(e) >= 300.  A masked key's score is
    // then raw - penalty (or - 2 penalty) <= -2^99 whenever |raw| < 2^98, so
    // 2^(x - m) underflows to exactly 0 however far its raw score lies above
    // the row's in-window scores; up to 2^125 two penalties still fit fp32.
    // (f16 masks in the softmax and does not use it.)
    {
        const int e = imax(100, int(ceilf(log2f(300.f / p.c_log2))));
        if (!f16 && e > 125) return ATTN_ERR_UNSUPPORTED;   // scale below ~1e-28
        p.penalty = ldexpf(1.f, imin(e, 125));
    }
    p.o = o;
    p.err = c.err;
    p.T = T; p.Hg = Hg; p.W = W;
    p.kt = kernel[0]; p.kh = kernel[1]; p.kw = kernel[2];
    p.et = imin(kernel[0], T); p.eh = imin(kernel[1], Hg); p.ew = imin(kernel[2], W);
    p.nbh = cdiv(Hg, p.bh);
    p.nbw = cdiv(W, p.bw);
    p.nbw2 = cdiv(p.nbw, 2);
    const dim3 grid(cdiv(T, p.bt) * p.nbh * p.nbw2, B * H);
    // the planner's key sub-box heights (4..8) have compile-time kernels (bf16)
    if (f16) return launch_tc<64, true, false, 0, true>(c, tq, tk, tv, p, grid);
    switch (p.KH) {
        case 4: return launch_tc<64, true, false, 4>(c, tq, tk, tv, p, grid);
        case 5: return launch_tc<64, true, false, 5>(c, tq, tk, tv, p, grid);
        case 6: return launch_tc<64, true, false, 6>(c, tq, tk, tv, p, grid);
        case 7: return launch_tc<64, true, false, 7>(c, tq, tk, tv, p, grid);
        case 8: return launch_tc<64, true, false, 8>(c, tq, tk, tv, p, grid);
        default: return launch_tc<64, true>(c, tq, tk, tv, p, grid);
    }
}

attn_status_t tc_selftest(const Ctx &c, const void *q, const void *k, const void *v,
                          const void *P, float *S, float *O, int D) {
    if (D != 64 && D != 128) return ATTN_ERR_UNSUPPORTED;
    CUtensorMap tq, tk, tv;
    const uint64_t dims[3] = {uint64_t(D), 128, 1};
    const uint32_t box[3] = {64, 128, 1};
    if (!make_tmap(&tq, q, 3, dims, box) || !make_tmap(&tk, k, 3, dims, box) ||
        !make_tmap(&tv, v, 3, dims, box))
        return ATTN_ERR_CUDA;
    const size_t smem = 3 * (D / 64) * 16384 + 8192 + 1024;
    static int done_mask = 0;
    if (D == 128) {
        if (!ensure_smem_attr(reinterpret_cast<const void *>(tc_selftest_kernel<128>), smem, c.device, &done_mask))
            return ATTN_ERR_RESOURCE;
        tc_selftest_kernel<128><<<1, 160, smem, c.stream>>>(
            tq, tk, tv, static_cast<const __nv_bfloat16 *>(q), static_cast<const __nv_bfloat16 *>(k),
            static_cast<const __nv_bfloat16 *>(P), S, O, c.err);
    } else {
        static int done64 = 0;
        if (!ensure_smem_attr(reinterpret_cast<const void *>(tc_selftest_kernel<64>), smem, c.device, &done64))
            return ATTN_ERR_RESOURCE;
        tc_selftest_kernel<64><<<1, 160, smem, c.stream>>>(
            tq, tk, tv, static_cast<const __nv_bfloat16 *>(q), static_cast<const __nv_bfloat16 *>(k),
            static_cast<const __nv_bfloat16 *>(P), S, O, c.err);
    }
    return launch_status(kFamTcFlash);
}

}  // namespace attn
