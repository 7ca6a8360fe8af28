// Tensor-core (tcgen05 + TMEM + TMA) flash attention for bf16 and f16, sm_103a:
// full attention (the joint text+image attention of FLUX) and causal
// grouped-query prefill.  (3D neighborhood attention has a persistent kernel
// of its own, tc_na.cu.)
//
// S = Q K^T * scale, row softmax, O = P V, streamed over key tiles with an
// online softmax (the attention of iris.c issue #15 "CUDA codepath !").  The
// page computes it as cuBLAS GEMM -> softmax kernel -> GEMM with S in HBM;
// here S and P never leave the SM.
//
// One CTA = two 128-row query tiles (Q0, Q1) of one (batch, head), 12 warps:
//   warps 0-3   softmax warpgroup of Q0 (thread = query row = TMEM lane)
//   warps 4-7   softmax warpgroup of Q1
//   warp  8     MMA issuer (one elected thread) and TMEM owner
//   warp  9     TMA loader of Q and the K ring (one elected thread)
//   warp 10     TMA loader of the V ring (one elected thread)
//   warp 11     barrier set-up, then idle
// The third warpgroup drops to 72 registers per thread (setmaxnreg) so the
// softmax warpgroups can hold a whole S row in registers (216 per thread).
//
// Key tiles of 128.  Tensor memory holds S_t at [128 t, 128 t + 128) and O_t
// at [256 + D t, 256 + D (t + 1)).  With D = 128 the columns are full and P_t
// (16-bit, two per column) overwrites the first 64 columns of S_t once the
// softmax has read S_t; with D = 64 P_t has columns of its own
// ([384 + 64 t, 448 + 64 t)).  One thread issues every MMA, per key tile j:
//   D = 128 (P over S):  PV0(j), QK0(j+1), PV1(j), QK1(j+1)   -- QK_t(j+1)
//       overwrites S_t only after PV_t(j) has read P_t (MMAs of one thread
//       execute in issue order);
//   D = 64 (separate P): QK0(j+1), QK1(j+1) as soon as the softmax has read
//       S_t(j) into registers, then PV0(j), PV1(j).
// The P V MMA takes P straight from TMEM (A operand) and V from shared memory
// (MN-major B operand).  K and V stream through rings of their own.
//
// Softmax (base 2): x = s * scale * log2(e).  The first tile sets the running
// max m; later tiles are exponentiated against m as it stands (no tile-max
// pass) and only a tile whose row sum overflows a bound is redone with its own
// max, which moves m if the tile max exceeds it by more than 8; only then is
// O_t rescaled in TMEM, after waiting for the previous PV_t to complete.
// Every branch that leads to a warp-collective tcgen05.ld / st is uniform
// across the warp.
//
// Both query tiles share each K/V tile.  Q, K and V are 4D tensor maps
// {D, N, heads, B} built from each tensor's element strides (contiguous for
// the plain entries), and the epilogue stores through the output's strides, so
// strided views are read and written in place.
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
constexpr int kBN = 128;      // keys per key tile (MMA N of S)

template <int D>
struct TcCfg {
    static constexpr int BN = kBN;                         // keys per key tile
    static constexpr int PANELS = D / 64;                  // 128-byte swizzle panels
    static constexpr int PANEL_Q = kBM * 128;              // bytes per Q panel
    static constexpr int PANEL_KV = BN * 128;              // bytes per K/V panel
    static constexpr int Q_BYTES = PANELS * PANEL_Q;
    static constexpr int KV_BYTES = PANELS * PANEL_KV;     // one K (or V) stage
    static constexpr int BUDGET = 227 * 1024 - 2048;
    static constexpr int NS_ALL = (BUDGET - kNQ * Q_BYTES) / KV_BYTES;
    // K and V rings of equal depth (a third K stage at D = 128 measured slower)
    static constexpr int KS = NS_ALL / 2 > 4 ? 4 : NS_ALL / 2;               // K stages
    static constexpr int VS = NS_ALL - NS_ALL / 2 > 4 ? 4 : NS_ALL - NS_ALL / 2;  // V stages
    static_assert(KS >= 2 && VS >= 2, "at least two K and two V stages");
    static constexpr int OFF_Q = 0;
    static constexpr int OFF_K = kNQ * Q_BYTES;
    static constexpr int OFF_V = OFF_K + KS * KV_BYTES;
    static constexpr int OFF_BAR = OFF_V + VS * KV_BYTES;
    static constexpr int SMEM = OFF_BAR + 512 + 1024;      // barriers + 1024 B alignment slack
    // Tensor memory (512 columns): S_t at t BN, O_t at kNQ BN + t D; P (16-bit,
    // two per column) over the first half of S_t (D = 128) or in columns of
    // its own after the O's (D = 64).
    static constexpr bool SEP_P = kNQ * (BN + D + BN / 2) <= 512;
    static constexpr uint32_t tm_s(int t) { return t * BN; }
    static constexpr uint32_t tm_o(int t) { return kNQ * BN + t * D; }
    static constexpr uint32_t tm_p(int t) { return SEP_P ? kNQ * BN + kNQ * D + t * (BN / 2) : t * BN; }
    static constexpr uint32_t TM_COLS = 512;
    static_assert(tm_o(kNQ - 1) + D <= TM_COLS && (!SEP_P || tm_p(kNQ) <= TM_COLS),
                  "tensor-memory layout must fit 512 columns");
    static constexpr int NSOFT = 4 * kNQ;
    static constexpr int W_MMA = NSOFT;                   // MMA issuer, TMEM owner
    static constexpr int W_LOAD = NSOFT + 1;              // Q and K copies
    static constexpr int W_LOADV = NSOFT + 2;             // V copies
    static constexpr int W_INIT = NSOFT + 3;              // barrier set-up
    static constexpr int NT = (NSOFT + 4) * 32;            // 3 warpgroups
    // register split: launch 168 x 384 = 64512; 2 x 128 x 216 + 128 x 72 = 64512
    static constexpr int REGS_LAUNCH = 168;
    static constexpr int REGS_SOFTMAX = 216;
    static constexpr int REGS_OTHER = 72;
    static_assert(2 * 128 * REGS_SOFTMAX + 128 * REGS_OTHER <= NT * REGS_LAUNCH,
                  "setmaxnreg split must fit the launch's register file share");
    static constexpr int k_off(int s) { return OFF_K + s * KV_BYTES; }
    static constexpr int v_off(int s) { return OFF_V + s * KV_BYTES; }
};

struct TcParams {
    int Nq, Nkv;             // query / key tokens per (batch, head)
    float c_log2;            // scale * log2(e)
    void *o;                 // bf16 or f16, like the inputs
    unsigned *err;
    // causal grouped-query prefill
    int Hq, Hkv, group;
    // q, k, v are 4D tensor maps {D, N, heads, B}; o is written through
    // element strides (batch, head, row), D contiguous
    int H;                   // query heads (the batch of block row bh is bh / H)
    long long o_sb, o_sh, o_sn;
};

// Barrier block at OFF_BAR.
template <int KS, int VS>
struct Bars {
    uint64_t q_full;
    // K and V rings are released separately: a K stage as soon as the Q K^T
    // products that read it have completed, a V stage after its P V
    uint64_t k_full[KS], k_empty[KS], v_full[VS], v_empty[VS];
    // per query tile t: s_full its Q K^T has completed, p_ready the softmax
    // has written P, o_done the P V product that read P has completed,
    // s_free (separate P, D = 64) the softmax holds S_t in registers
    uint64_t s_full[kNQ], p_ready[kNQ], o_done[kNQ], s_free[kNQ];
    uint64_t drain;
    uint32_t tmem_base;
    int abort;
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

// CAUSAL: grouped-query causal prefill (query tile t sees key tiles up to its
// diagonal).  F16: inputs, P and output in f16 instead of bf16 (same layouts;
// the MMA operand format flips).
template <int D, bool CAUSAL, bool F16>
__global__ void __launch_bounds__(TcCfg<D>::NT, 1)
tc_attn_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
               const __grid_constant__ CUtensorMap tv, const TcParams p) {
    using C = TcCfg<D>;
    using BarsT = Bars<C::KS, C::VS>;
    static_assert(sizeof(BarsT) <= 512, "barrier block must fit its reserved bytes");
    extern __shared__ uint8_t smem_raw[];
    // 1024-byte alignment for the 128-byte swizzle atoms
    uint8_t *smem = smem_raw + ((1024 - (ptx::smem_addr(smem_raw) & 1023)) & 1023);
    BarsT *bars = reinterpret_cast<BarsT *>(smem + C::OFF_BAR);
    volatile int *abort = &bars->abort;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int bh = blockIdx.y;
    // batch and head of this block row, and the K/V head (the query head's KV
    // head for grouped-query attention: contiguous groups of Hq / Hkv heads)
    const int fb = bh / p.H, fh = bh % p.H;
    const int fkh = CAUSAL ? fh / p.group : fh;

    // ---- per-CTA work description (identical in every role)
    int n_t[kNQ];
    int steps;
    int q0;
    constexpr int BNt = C::BN;     // keys per tile
    if constexpr (CAUSAL) {
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

    if (warp == C::W_INIT && lane == 0) {
        ptx::mbar_init(&bars->q_full, 1);
        for (int s = 0; s < C::KS; ++s) {
            ptx::mbar_init(&bars->k_full[s], 1);
            ptx::mbar_init(&bars->k_empty[s], 1);
        }
        for (int s = 0; s < C::VS; ++s) {
            ptx::mbar_init(&bars->v_full[s], 1);
            ptx::mbar_init(&bars->v_empty[s], 1);
        }
        for (int t = 0; t < kNQ; ++t) {
            ptx::mbar_init(&bars->s_full[t], 1);
            ptx::mbar_init(&bars->p_ready[t], 128);
            ptx::mbar_init(&bars->o_done[t], 1);
            ptx::mbar_init(&bars->s_free[t], 128);
        }
        ptx::mbar_init(&bars->drain, 1);
        bars->abort = 0;
        ptx::fence_barrier_init();
    }
    if (warp == C::W_MMA) {
        ptx::tmem_alloc(&bars->tmem_base, C::TM_COLS);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = bars->tmem_base;
    // launched as a programmatic dependent of the previous kernel (the RoPE
    // pass writes this kernel's Q and K): the set-up above touches nothing
    // global, the copies below wait for that kernel to complete; a decode
    // launched behind this kernel may start launching at once
    ptx::griddep_wait();
    ptx::griddep_launch_dependents();

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
                ptx::mbar_arrive_expect_tx(&bars->q_full, kNQ * C::Q_BYTES);
#pragma unroll
                for (int t = 0; t < kNQ; ++t)
                    for (int pn = 0; pn < C::PANELS; ++pn)
                        ptx::tma_load_4d(smem + C::OFF_Q + t * C::Q_BYTES + pn * C::PANEL_Q, &tq, pn * 64,
                                         q0 + t * kBM, fh, fb, &bars->q_full, pol_q);
            }
            const int NS = which == 0 ? C::KS : C::VS;   // depth of this ring
            int issued = 0;
            for (int j = 0; j < steps; ++j) {
                const int s = j % NS;
                if (j >= NS && !ptx::mbar_wait_or_abort(&empty[s], ((j / NS) - 1) & 1, p.err, abort))
                    break;
                issued = j + 1;
                // the K/V stream serves both query tiles, so it runs for the
                // longer of the two tile counts
                ptx::mbar_arrive_expect_tx(&full[s], C::KV_BYTES);
                for (int pn = 0; pn < C::PANELS; ++pn)
                    ptx::tma_load_4d(smem + (which == 0 ? C::k_off(s) : C::v_off(s)) + pn * C::PANEL_KV, tm,
                                     pn * 64, j * kBN, fkh, fb, &full[s], pol_kv);
            }
            // after a timeout elsewhere: let the copies this thread issued land
            // (bounded) before the CTA's shared memory is released
            if (*abort) {
                if (which == 0) ptx::mbar_wait(&bars->q_full, 0, nullptr);
                for (int j = imax(0, issued - NS); j < issued; ++j)
                    ptx::mbar_wait(&full[j % NS], (j / NS) & 1, nullptr);
            }
        } else if (warp == C::W_MMA && lane == 0) {
            // ============================================= MMA issuer
            const uint32_t id_qk = ptx::idesc_16_f32(kBM, BNt, false, F16);
            const uint32_t id_pv = ptx::idesc_16_f32(kBM, D, true, F16);
            // Matrix descriptors are built once: a k-step, a stage or a tile only
            // moves the start-address field (bits 0-13, byte address >> 4, no
            // carry out of it below 256 KB), so each MMA costs one add here
            // instead of a rebuilt 64-bit descriptor on this single thread.
            constexpr uint32_t HI128 = ptx::desc_hi_sw128(1024);
            const uint32_t dq0 = ptx::desc_lo_sw128(ptx::smem_addr(smem + C::OFF_Q), 16);
            const uint32_t dk0 = ptx::desc_lo_sw128(ptx::smem_addr(smem + C::k_off(0)), 16);
            const uint32_t dv0 = ptx::desc_lo_sw128(ptx::smem_addr(smem + C::v_off(0)), C::PANEL_KV);
            constexpr int nkv = BNt / 16;        // k-steps of P V
            auto issue_qk = [&](int t, int j) {
                const uint32_t a0 = dq0 + uint32_t((t * C::Q_BYTES) >> 4);
                const uint32_t b0 = dk0 + uint32_t(((j % C::KS) * C::KV_BYTES) >> 4);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t oa = ((kk >> 2) * C::PANEL_Q + (kk & 3) * 32) >> 4;
                    const uint32_t ob = ((kk >> 2) * C::PANEL_KV + (kk & 3) * 32) >> 4;
                    ptx::mma_ss(tmem + C::tm_s(t), ptx::desc_join(a0 + oa, HI128),
                                ptx::desc_join(b0 + ob, HI128), id_qk, kk > 0);
                }
                ptx::tc_commit(&bars->s_full[t]);
            };
            auto issue_pv = [&](int t, int j) {
                const uint32_t b0 = dv0 + uint32_t(((j % C::VS) * C::KV_BYTES) >> 4);
                const uint32_t a0 = tmem + C::tm_p(t);
#pragma unroll
                for (int kk = 0; kk < nkv; ++kk)
                    ptx::mma_ts(tmem + C::tm_o(t), a0 + kk * 8,
                                ptx::desc_join(b0 + uint32_t(kk * (2048 >> 4)), HI128), id_pv,
                                (j > 0 || kk > 0) ? 1u : 0u);
                ptx::tc_commit(&bars->o_done[t]);
            };
            bool ok = ptx::mbar_wait_or_abort(&bars->q_full, 0, p.err, abort) &&
                      (steps == 0 || ptx::mbar_wait_or_abort(&bars->k_full[0], 0, p.err, abort));
            ptx::tc_fence_after();
            // Each stage barrier is waited on once per use (a completed wait
            // still costs this thread a round trip to shared memory).
            bool k_seen = false, v_seen = false;
            auto wait_k = [&](int jn) {
                if (!k_seen) {
                    ok = ok && ptx::mbar_wait_or_abort(&bars->k_full[jn % C::KS], (jn / C::KS) & 1, p.err, abort);
                    k_seen = true;
                }
            };
            auto wait_v = [&](int j) {
                if (!v_seen) {
                    ok = ok && ptx::mbar_wait_or_abort(&bars->v_full[j % C::VS], (j / C::VS) & 1, p.err, abort);
                    v_seen = true;
                }
            };
            // Q K^T of key tile jn for tile t, once the softmax no longer needs
            // the S it overwrites (separate P: as soon as the softmax holds
            // S(jprev) in registers; P over S: after P V (jprev), issued before)
            auto next_qk = [&](int t, int jn, int jprev) {
                if (jn < pick(n_t, t)) {
                    if (C::SEP_P)
                        ok = ok && ptx::mbar_wait_or_abort(&bars->s_free[t], jprev & 1, p.err, abort);
                    wait_k(jn);
                    if (!ok) return;
                    ptx::tc_fence_after();
                    issue_qk(t, jn);
                } else {
                    wait_k(jn);
                }
            };
            // P V of key tile j for tile t
            auto this_pv = [&](int t, int j) {
                if (j < pick(n_t, t)) {
                    ok = ok && ptx::mbar_wait_or_abort(&bars->p_ready[t], j & 1, p.err, abort);
                    wait_v(j);
                    if (!ok) return;
                    ptx::tc_fence_after();
                    issue_pv(t, j);
                } else {
                    wait_v(j);
                }
            };
            if (ok) {
#pragma unroll
                for (int t = 0; t < kNQ; ++t)
                    if (n_t[t] > 0) issue_qk(t, 0);
                if (steps > 0) ptx::tc_commit(&bars->k_empty[0]);
            }
            for (int j = 0; ok && j < steps; ++j) {
                const int jn = j + 1;
                k_seen = v_seen = false;
                if constexpr (C::SEP_P) {
                    // separate P: the next S as soon as the softmax holds the
                    // current one in registers, then P V
#pragma unroll
                    for (int t = 0; t < kNQ; ++t)
                        if (ok && jn < steps) next_qk(t, jn, j);
#pragma unroll
                    for (int t = 0; t < kNQ; ++t)
                        if (ok) this_pv(t, j);
                } else {
                    // P over S: the Q K^T that overwrites S_t follows the P V that
                    // reads P there (one thread's MMAs execute in issue order)
#pragma unroll
                    for (int t = 0; t < kNQ; ++t) {
                        if (ok) this_pv(t, j);
                        if (ok && jn < steps) next_qk(t, jn, j);
                    }
                }
                if (!ok) break;
                // Q K^T of key tile j + 1 and P V of key tile j are issued
                if (jn < steps) ptx::tc_commit(&bars->k_empty[jn % C::KS]);
                ptx::tc_commit(&bars->v_empty[j % C::VS]);
            }
            // drain: every MMA has completed before TMEM is freed
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
        const uint32_t o_addr = lane_base + C::tm_o(t);
        const uint32_t s_addr = lane_base + C::tm_s(t);
        const uint32_t p_addr = lane_base + C::tm_p(t);
        const float cl = p.c_log2;
        const int nt = pick(n_t, t);
        const bool qvalid = q0 + t * kBM + row < p.Nq;

        // waits for the P V product of key tile jj of this query tile (and so
        // for every earlier one: one thread's MMAs complete in issue order)
        auto wait_pv = [&](int jj) -> bool {
            if (!__all_sync(0xffffffffu, ptx::mbar_wait_or_abort(&bars->o_done[t], jj & 1, p.err, abort)))
                return false;
            ptx::tc_fence_after();
            return true;
        };

        float m = -INFINITY, l = 0.f;
        bool ok = true;
        for (int j = 0; j < nt; ++j) {
            if (!__all_sync(0xffffffffu, ptx::mbar_wait_or_abort(&bars->s_full[t], j & 1, p.err, abort))) {
                ok = false;
                break;
            }
            ptx::tc_fence_after();

            float sv[BNt];
#pragma unroll
            for (int c = 0; c < BNt / 32; ++c)
                ptx::tmem_ld32(s_addr + c * 32, *reinterpret_cast<uint32_t(*)[32]>(&sv[c * 32]));
            ptx::tmem_wait_ld();
            if constexpr (C::SEP_P) {
                // S_t is in registers: the next QK_t may overwrite it
                ptx::tc_fence_before();
                ptx::mbar_arrive(&bars->s_free[t]);
            }

            // ---- masks: keys past the sequence; causal: the last tile is the
            //      diagonal one (query tile and key tile start at the same
            //      position), key e is visible to row `row` iff e <= row
            {
                int valid = p.Nkv - j * BNt;
                if constexpr (CAUSAL) {
                    if (j == nt - 1) {
#pragma unroll
                        for (int e = 0; e < BNt; ++e)
                            if (e > row || e >= valid) sv[e] = -INFINITY;
                        valid = BNt;
                    }
                }
                if (valid < BNt) {
#pragma unroll
                    for (int e = 0; e < BNt; ++e)
                        if (e >= valid) sv[e] = -INFINITY;
                }
            }

            // P = 2^(x - m) in 16-bit into TMEM; returns the tile's row sum (fp32)
            auto emit_p = [&](float nmu) -> float {
                float acc[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) acc[i] = 0.f;
#pragma unroll
                for (int c = 0; c < BNt / 32; ++c) {
                    uint32_t pk[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        float x0, x1;
                        ptx::ffma2(x0, x1, sv[c * 32 + 2 * e], sv[c * 32 + 2 * e + 1], cl, cl, nmu, nmu);
                        const float p0 = ptx::ex2(x0), p1 = ptx::ex2(x1);
                        ptx::fadd2(acc[(2 * e) & 7], acc[(2 * e + 1) & 7], acc[(2 * e) & 7],
                                   acc[(2 * e + 1) & 7], p0, p1);
                        pk[e] = H16<F16>::pack(p0, p1);
                    }
                    ptx::tmem_st16(p_addr + c * 16, pk);
                }
                return ((acc[0] + acc[1]) + (acc[2] + acc[3])) + ((acc[4] + acc[5]) + (acc[6] + acc[7]));
            };

            // ---- P in columns of its own: the P V product that last read them
            //      (key tile j - 1) must be done.  P over S needs no wait: the
            //      Q K^T that wrote this S was issued after the P V that read the
            //      P last held here, and MMAs complete in issue order.
            bool prev_done = false;              // P V of tile j - 1 observed complete
            if (C::SEP_P && j >= 1) {
                if (!wait_pv(j - 1)) {
                    ok = false;
                    break;
                }
                prev_done = true;
            }

            // ---- fast path: exponentiate against the running maximum m as it
            //      stands, with no tile maximum.  P only has to stay finite in its
            //      16-bit type, not below 1: a tile whose row sum exceeds 2^24 (2^15
            //      for f16, whose largest finite value is 65504) or is not finite
            //      is redone below against its own maximum.  After the first tiles
            //      m is close to the row maximum and the redo almost never runs.
            bool fast = j > 0 && __all_sync(0xffffffffu, m != -INFINITY);
            if (fast) {
                const float lt = emit_p(-m);
                if (__any_sync(0xffffffffu, !(lt <= (F16 ? 32768.f : 16777216.f))))
                    fast = false;                 // redo the tile (P is rewritten below)
                else
                    l += lt;
            }

            if (!fast) {
                // ---- tile maximum
                float mx[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) mx[i] = -INFINITY;
#pragma unroll
                for (int e = 0; e < BNt; e += 8) {
#pragma unroll
                    for (int i = 0; i < 8; ++i) mx[i] = fmaxf(mx[i], sv[e + i]);
                }
                const float tmax = fmaxf(ptx::fmax3(ptx::fmax3(mx[0], mx[1], mx[2]), ptx::fmax3(mx[3], mx[4], mx[5]),
                                                    mx[6]),
                                         mx[7]);
                const float mt = tmax * cl;      // cl > 0: max commutes with the scaling

                // ---- the previous P V must be done before O is rescaled
                const bool want = j == 0 || mt > m + 8.f;   // this row moves its maximum
                const bool any_want = __any_sync(0xffffffffu, want);
                if (j > 0 && any_want && !prev_done) {
                    if (!wait_pv(j - 1)) {
                        ok = false;
                        break;
                    }
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
                l += emit_p((m == -INFINITY) ? 0.f : -m);
            }
            ptx::tmem_wait_st();
            ptx::tc_fence_before();
            ptx::mbar_arrive(&bars->p_ready[t]);
        }

        // ---- epilogue: O / l -> 16-bit -> global
        if (ok && nt > 0 && wait_pv(nt - 1)) {
            const float inv = 1.f / l;
            typename H16<F16>::T *orow = nullptr;
            if (qvalid)
                orow = static_cast<typename H16<F16>::T *>(p.o) +
                       size_t(fb * p.o_sb + fh * p.o_sh + (long long)(q0 + t * kBM + row) * p.o_sn);
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

template <int D, bool CAUSAL = false, bool F16 = false>
attn_status_t launch_tc(const Ctx &c, const CUtensorMap &tq, const CUtensorMap &tk,
                        const CUtensorMap &tv, const TcParams &p, dim3 grid) {
    using C = TcCfg<D>;
    static int done_mask = 0;
    static int regs = -1;
    auto kern = tc_attn_kernel<D, CAUSAL, F16>;
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
    // programmatic dependent launch: the CTAs set up while the previous
    // kernel finishes and wait for it before their first copy
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(C::NT);
    cfg.dynamicSmemBytes = C::SMEM;
    cfg.stream = c.stream;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, kern, tq, tk, tv, p) != cudaSuccess) {
        cudaGetLastError();
        return ATTN_ERR_CUDA;
    }
    return launch_status(kFamTcFlash);
}

}  // namespace

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

bool make_tmap(CUtensorMap *m, const void *base, int rank, const uint64_t *dims,
               const uint32_t *box, bool f16) {
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

bool tma_encode_available() { return encode_fn() != nullptr; }

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
        return D == 128 ? launch_tc<128, false, true>(c, tq, tk, tv, p, grid)
                        : launch_tc<64, false, true>(c, tq, tk, tv, p, grid);
    return D == 128 ? launch_tc<128>(c, tq, tk, tv, p, grid) : launch_tc<64>(c, tq, tk, tv, p, grid);
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
        return D == 128 ? launch_tc<128, true, true>(c, tq, tk, tv, p, grid)
                        : launch_tc<64, true, true>(c, tq, tk, tv, p, grid);
    return D == 128 ? launch_tc<128, true>(c, tq, tk, tv, p, grid) : launch_tc<64, true>(c, tq, tk, tv, p, grid);
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
