// Persistent tensor-core (tcgen05 + TMEM + TMA) 3D neighborhood attention for
// bf16 and f16, sm_103a: the neighborhood attention of candle PR #11 ("3D
// neighborhood attention", NATTEN boundary windows: window start
// clamp(i - k/2, 0, n - k_eff) per axis), computed as a fused flash-style
// kernel whose scores never leave the SM.
//
// Each CTA (one per SM) runs two independent query-tile streams: stream t
// of CTA c takes the 3D query boxes (<= 128 queries each, w fastest, then h,
// t, batch x head) 2c + t, 2c + t + 2 grid, ... (the last, partial round
// spread one box per CTA), so the CTAs in flight hold
// neighbouring boxes of one head (their key windows overlap in L2), and the
// set-up that a CTA per box paid every time (barriers, tensor memory, the
// query-offset channels, the first copies and the first Q K^T) is paid once
// or hidden behind the previous box: a stream's loader streams the next box's
// key tiles as soon as its ring stages free up, the next box's queries load
// once the last Q K^T of the current one has completed, and its first two
// Q K^T are issued while the softmax warps are still writing out the current
// box's outputs.  A box change still idles a stream's issuer for the length
// of the epilogue and the next box's first softmax, so stream 1 starts about
// half a box late: the two streams change boxes at different times, and
// while one changes the other has the tensor pipe to itself.
//
// Per box the keys are the union of the box's clamped windows (a 3D box
// again, the window start being monotone), streamed as (KT, KH, 16) key
// sub-boxes of 96 keys by 5D TMA into each stream's own K and V rings.
// bf16 applies the h and w window tests on the tensor core.  Measured from
// the union's origin, a query's h window is [a, a + eh) and its w window
// [b, b + ew), with a < bh and b < bw (the clamped window start advances by
// 0 or 1 per row); every query row carries 16 one-hot channels (channel a and
// channel bh + b) and every key sub-box 16 channels holding -2^100 (at least;
// see the host) where the key's union row / column lies outside the window of
// that offset.  One extra 16-deep MMA step thus adds -2^100 per violated axis
// to S, and every masked key gets P = 0 exactly whenever the raw scores are
// below 2^98 in magnitude.  The key side depends only on the sub-box's place
// in the union, not on the box, so its channel tiles are built once per CTA;
// a softmax thread writes its own row's query channels for each box.  f16
// cannot hold such a penalty and tests h and w per key in the softmax.  The t
// window is tested per 16-key group (one frame of the sub-box).
//
// Warps: 0-3 softmax of stream 0 (thread = query row = TMEM lane), 4-7 of
// stream 1, 8 MMA issuer of stream 0 and TMEM owner, 9 and 10 TMA loaders of
// stream 0 and 1 (Q, K and V in the order the issuer consumes them), 11 MMA
// issuer of stream 1 (and barrier set-up).  The third warpgroup drops to 72
// registers (setmaxnreg) so the softmax warpgroups hold a whole score row in
// registers (216).
//
// Tensor memory per stream t: [S_t,0 | S_t,1 | O_t] (96 + 96 + 64 columns)
// at 256 t.  Key tile g of the stream (counted over all its boxes) has its
// scores in buffer g % 2, and its P is written over them; the issuer of
// stream t issues P V (g) as soon as the softmax has written P(g) and right
// behind it Q K^T (g + 2) into the same buffer (one thread's MMAs execute in
// order), so the next scores are ready when the softmax finishes a key tile.
// Every barrier is waited for phase by phase, never skipping one, and each is
// at most one phase ahead of any waiter (argued per barrier below): a parity
// wait cannot tell phase k from phase k + 2.
//
// Softmax (base 2): x = s * scale * log2(e); the first key tile sets the
// running max m, later tiles are exponentiated against m as it stands and a
// tile whose row sum overflows a bound (or is not finite) is redone with its
// own max, moving m (and rescaling O in TMEM after the previous P V) only
// when the tile max exceeds it by more than 8.  32-key chunks outside the t
// window of all 32 rows of a warp are written as P = 0 without exponentials.
//
// All spin-waits are bounded (1 s); on a timeout the CTA raises the device
// error word, lets the copies it issued land, frees TMEM and exits.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "common.cuh"
#include "kernels.h"
#include "ptx.cuh"

namespace attn {
namespace {

constexpr int kBM = 128;            // query rows per tile (MMA M)
constexpr int kNQ = 2;              // query-tile streams per CTA
constexpr int kBN = 96;             // keys per key tile: a (KT, KH, 16) sub-box, KT KH = 6
constexpr int kD = 64;              // head dimension
constexpr int kKW = 16;             // key sub-box width along w
constexpr int kMaxPenaltyTiles = 7; // key penalty tiles: union h chunks x w chunks

template <bool PEN>
struct NaCfg {
    static constexpr int PANEL = kBM * 128;              // one query tile (64 channels, 128 B rows)
    static constexpr int KV_BYTES = kBN * 128;           // one K or V tile
    static constexpr int STAGE_BYTES = kNQ * KV_BYTES;   // stage s of both streams' rings
    // window channels: 16 16-bit values per row, 32-byte swizzle
    static constexpr int X_ROW = 32;
    static constexpr int MAXV = PEN ? kMaxPenaltyTiles : 0;
    static constexpr int QX_BYTES = PEN ? kNQ * kBM * X_ROW : 0;   // query channels per stream
    static constexpr int KX_BYTES = kBN * X_ROW;         // one key penalty tile
    static constexpr int KXV_BYTES = MAXV * KX_BYTES;    // shared by both streams
    static constexpr int BUDGET = 227 * 1024 - 1536;      // all but the barrier block and alignment slack
    static constexpr int OFF_Q = 0;
    static constexpr int OFF_QX = OFF_Q + kNQ * PANEL;
    static constexpr int OFF_KXV = OFF_QX + QX_BYTES;
    static constexpr int OFF_K = (OFF_KXV + KXV_BYTES + 1023) / 1024 * 1024;   // 128-byte swizzle atoms
    static constexpr int NS_ALL = (BUDGET - OFF_K) / STAGE_BYTES;
    // V gets the deeper ring: the K tile of step g + 2 and the V tile of
    // step g are read by the same issuer step, so with K 2 / V 4 stages one
    // completion (Q K^T (g)) frees both stages that tile g + 2 refills.
    // Measured on the large workload (with rings shared by both query tiles
    // and separate stage releases): K 2 / V 4 stages 944.7 us, K 3 / V 3
    // 946.8, K 3 / V 2 (before the query channels were shared) 966.0, K 2 /
    // V 3 953.1.
    static constexpr int VS = NS_ALL - 2 > 4 ? 4 : NS_ALL - 2;
    static constexpr int KS = NS_ALL - VS > 4 ? 4 : NS_ALL - VS;
    static_assert(KS >= 2 && VS >= 4, "Q K^T (g) must free the K and V stages of tile g + 2");
    static constexpr int OFF_V = OFF_K + KS * STAGE_BYTES;
    static constexpr int OFF_BAR = OFF_V + VS * STAGE_BYTES;
    static constexpr int SMEM = OFF_BAR + 512 + 1024;    // barriers + 1024 B alignment slack
    static_assert(SMEM <= 227 * 1024, "shared memory of one CTA");
    // tensor memory
    static constexpr uint32_t tm_s(int t, int b) { return t * 256 + b * kBN; }
    static constexpr uint32_t tm_o(int t) { return t * 256 + 2 * kBN; }
    static constexpr uint32_t TM_COLS = 512;
    static_assert(tm_o(kNQ - 1) + kD <= TM_COLS, "tensor-memory layout must fit 512 columns");
    // warps
    static constexpr int NSOFT = 4 * kNQ;
    static constexpr int W_MMA = NSOFT;       // issuer of stream 0, TMEM owner
    static constexpr int W_LOAD = NSOFT + 1;  // Q, K and V copies of stream 0
    static constexpr int W_LOAD1 = NSOFT + 2; // Q, K and V copies of stream 1
    static constexpr int W_MMA1 = NSOFT + 3;  // issuer of stream 1, barrier set-up
    static constexpr int NT = (NSOFT + 4) * 32;
    // threads that zero the query rows past the box and build the key penalty tiles
    static constexpr int NBUILD = NT - 32;
    // register split: launch 168 x 384 = 64512 = 2 x 128 x 216 + 128 x 72
    static constexpr int REGS_LAUNCH = 168;
    static constexpr int REGS_SOFTMAX = 216;
    static constexpr int REGS_OTHER = 72;
    static_assert(2 * 128 * REGS_SOFTMAX + 128 * REGS_OTHER <= NT * REGS_LAUNCH,
                  "setmaxnreg split must fit the launch's register file share");
    static constexpr int k_off(int s, int u) { return OFF_K + s * STAGE_BYTES + u * KV_BYTES; }
    static constexpr int v_off(int s, int u) { return OFF_V + s * STAGE_BYTES + u * KV_BYTES; }
    static constexpr int qx_off(int u) { return OFF_QX + u * kBM * X_ROW; }
    static constexpr int kxv_off(int v) { return OFF_KXV + v * KX_BYTES; }
};

struct NaParams {
    float c_log2;            // scale * log2(e)
    float penalty;           // bf16: power of two >= 2^100 with penalty * c_log2 >= 300
    void *o;                 // [B * heads, T * Hg * W, 64], like the inputs
    unsigned *err;
    int T, Hg, W;            // grid (row-major)
    int kt, kh, kw;          // requested kernel
    int et, eh, ew;          // effective kernel (min(k, extent))
    int bt, bh, bw;          // query box
    int nbt, nbh, nbw;       // boxes along t, h, w
    int KT, KH;              // key sub-box frames and rows (KT KH 16 = 96 keys)
    int nhv, nwv;            // most union h / w chunks of a box (penalty tiles nhv nwv)
    int n_boxes;             // boxes x (batch x heads)
    int stagger;             // stream 1 starts once stream 0 has issued this many P V
};

// Barrier block at OFF_BAR.  Phases (k counts from 0) of stream t's barriers:
//   q_full [t] k: the queries and the first two K tiles of the stream's box k
//                  have landed
//   q_free [t] k: every Q K^T of box k has completed
//   s_full [2 t + b]: Q K^T of the stream's key tile g (g % 2 = b) has completed;
//                  this also frees the K and V stages of tile g + 2: the K
//                  stage last held tile g + 2 - KS (KS >= 2), read by a Q K^T
//                  issued no later than Q K^T (g), and the V stage tile
//                  g + 2 - VS (VS >= 4), read by a P V issued before it (the
//                  issuer puts P V (g - 2) before Q K^T (g))
//   ready [t][g % 4]: the issuer's key-tile step g may run: the softmax has
//                  written P(g) (128 arrivals), V(g) has landed and K(g + 2)
//                  has landed (one loader arrival with its bytes each; a plain
//                  one where tile g + 2 is not in the same box, as its K
//                  counts on its own box's q_full).  Every arrival of
//                  step g comes after step g - 4 has run (P(g) and the copies
//                  follow Q K^T (g - 2) or (g), issued at step g - 4 or later),
//                  and the issuer waits for step g before it issues the
//                  Q K^T (g + 2) that step g + 4 needs
//   o_done [2 t + b]: P V (g) has completed
//   chan_ready[t] k: the query channels of the stream's box k are written
//                  (128 arrivals)
//   go: stream 1 may start (one phase, one arrival from issuer 0)
struct NaBars {
    uint64_t q_full[kNQ], q_free[kNQ];
    uint64_t ready[kNQ][4];
    uint64_t s_full[2 * kNQ], o_done[2 * kNQ];
    uint64_t chan_ready[kNQ];
    uint64_t go;
    uint64_t drain;
    uint32_t tmem_base;
    int abort;
};

// One query box and the union of its windows.
struct NaTile {
    int t0, h0, w0;          // box origin
    int u0t, u0h, u0w;       // union origin
    int ntc, nhc, nwc;       // union chunks along t, h, w (KT frames, KH rows, 16 columns)
    int ntiles;              // key tiles = ntc nhc nwc
};

__host__ __device__ __forceinline__ NaTile na_tile(const NaParams &p, int bi_t, int bi_h, int bi_w,
                                                   int KT, int KH) {
    NaTile g;
    g.t0 = bi_t * p.bt;
    g.h0 = bi_h * p.bh;
    g.w0 = bi_w * p.bw;
    const int t1 = imin(g.t0 + p.bt, p.T) - 1, h1 = imin(g.h0 + p.bh, p.Hg) - 1,
              w1 = imin(g.w0 + p.bw, p.W) - 1;
    g.u0t = na_window_start(g.t0, p.T, p.kt);
    g.u0h = na_window_start(g.h0, p.Hg, p.kh);
    g.u0w = na_window_start(g.w0, p.W, p.kw);
    const int ut = na_window_start(t1, p.T, p.kt) + p.et - g.u0t;
    const int uh = na_window_start(h1, p.Hg, p.kh) + p.eh - g.u0h;
    const int uw = na_window_start(w1, p.W, p.kw) + p.ew - g.u0w;
    g.ntc = cdiv(ut, KT);
    g.nhc = cdiv(uh, KH);
    g.nwc = cdiv(uw, kKW);
    g.ntiles = g.ntc * g.nhc * g.nwc;
    return g;
}

// Box b: (batch x head) b / boxes, then box t, h, w (w fastest).
struct NaBox {
    NaTile g;
    int bhd;                 // batch x head
};

__device__ __forceinline__ NaBox na_box(const NaParams &p, int b, int KT, int KH) {
    NaBox x;
    const int per = p.nbt * p.nbh * p.nbw;
    x.bhd = b / per;
    const int r = b - x.bhd * per;
    x.g = na_tile(p, r / (p.nbh * p.nbw), (r / p.nbw) % p.nbh, r % p.nbw, KT, KH);
    return x;
}

// Box k of stream t of CTA c (-1 past the stream's last): the full rounds of
// 2 grid boxes go out in order (stream t of CTA c takes box 2c + t of each),
// and the boxes of the last, partial round one per CTA first (stream 0 of
// CTAs 0, 1, ..., then stream 1), so no CTA gets two boxes more than another
// and a CTA's extra box runs while its other stream is idle.
__device__ __forceinline__ int na_stream_box(const NaParams &p, int t, int k) {
    const int S = 2 * int(gridDim.x), K = p.n_boxes / S;
    if (k < K) return k * S + 2 * int(blockIdx.x) + t;
    const int i = t * int(gridDim.x) + int(blockIdx.x);
    return (k == K && i < p.n_boxes - K * S) ? K * S + i : -1;
}

// Origin (t, h, w) of key sub-box j of a tile: w chunk fastest, then h, then t.
__device__ __forceinline__ void na_key_box(const NaTile &g, int KT, int KH, int j, int &t, int &h,
                                           int &w) {
    const int wc = j % g.nwc;
    const int hc = (j / g.nwc) % g.nhc;
    const int tc = j / (g.nwc * g.nhc);
    t = g.u0t + tc * KT;
    h = g.u0h + hc * KH;
    w = g.u0w + wc * kKW;
}

// KSH = 10 KT + KH > 0 fixes the key sub-box at compile time (the softmax's
// group masks unroll); 0 takes KT and KH from the parameters.  F16: inputs, P
// and output in f16 (window tests in the softmax instead of penalty channels).
template <int KSH, bool F16>
__global__ void __launch_bounds__(NaCfg<!F16>::NT, 1)
tc_na_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
             const __grid_constant__ CUtensorMap tv, const NaParams p) {
    constexpr bool PEN = !F16;
    using C = NaCfg<PEN>;
    using BarsT = NaBars;
    static_assert(sizeof(BarsT) <= 512, "barrier block must fit its reserved bytes");
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024 - (ptx::smem_addr(smem_raw) & 1023)) & 1023);
    BarsT *bars = reinterpret_cast<BarsT *>(smem + C::OFF_BAR);
    volatile int *abort = &bars->abort;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int KT = KSH > 0 ? KSH / 10 : p.KT;
    const int KH = KSH > 0 ? KSH % 10 : p.KH;
    const int rows = p.bt * p.bh * p.bw;          // queries per box (<= 128)
    // a kernel launched behind this one as a programmatic dependent (decode)
    // may take the SMs this grid's CTAs leave; it waits for this grid to
    // complete before it reads anything
    ptx::griddep_launch_dependents();

    // ---- set-up: barriers (one thread of the last warp) beside the zero
    //      query rows past the box and the key penalty tiles, which are the
    //      same for every box (the other threads)
    if (threadIdx.x == C::NT - 32) {
        for (int t = 0; t < kNQ; ++t) {
            ptx::mbar_init(&bars->q_full[t], 1);
            ptx::mbar_init(&bars->q_free[t], 1);
            for (int s = 0; s < 4; ++s) ptx::mbar_init(&bars->ready[t][s], 128 + 2);
        }
        for (int b = 0; b < 2 * kNQ; ++b) {
            ptx::mbar_init(&bars->s_full[b], 1);
            ptx::mbar_init(&bars->o_done[b], 1);
        }
        for (int t = 0; t < kNQ; ++t) ptx::mbar_init(&bars->chan_ready[t], 128);
        ptx::mbar_init(&bars->go, 1);
        ptx::mbar_init(&bars->drain, kNQ);
        bars->abort = 0;
        ptx::fence_barrier_init();
    } else if (threadIdx.x < C::NBUILD) {
        // query rows past the box hold zeros (TMA writes the box's rows only)
        for (int i = threadIdx.x; i < kNQ * (kBM - rows) * 8; i += C::NBUILD) {
            const int chunk = i % 8, r = rows + (i / 8) % (kBM - rows), t = i / (8 * (kBM - rows));
            *reinterpret_cast<uint4 *>(smem + C::OFF_Q + t * C::PANEL + r * 128 + chunk * 16) =
                make_uint4(0, 0, 0, 0);
        }
        if constexpr (PEN) {
            // key penalty tile v = hc nwv + wc (union h chunk hc, w chunk wc):
            // key r lies on union row hc KH + (r / 16) % KH and column
            // wc 16 + r % 16 (the same in each of its KT frames); channel
            // c < bh holds -penalty where that row is outside [c, c + eh),
            // channel bh + c where the column is outside [c, c + ew)
            const typename H16<F16>::T negh = H16<F16>::from(-p.penalty);
            const uint32_t neg = uint32_t(*reinterpret_cast<const uint16_t *>(&negh));
            for (int i = threadIdx.x; i < p.nhv * p.nwv * kBN * 2; i += C::NBUILD) {
                const int half = i & 1, r = (i >> 1) % kBN, v = (i >> 1) / kBN;
                const int hc = v / p.nwv, wc = v - hc * p.nwv;
                const int uh = hc * KH + (r / kKW) % KH, uw = wc * kKW + r % kKW;
                uint32_t bits = 0u;
                for (int c = 0; c < 8; ++c) {
                    const int ch = half * 8 + c;
                    const bool out = ch < p.bh ? unsigned(uh - ch) >= unsigned(p.eh)
                                   : ch < p.bh + p.bw ? unsigned(uw - (ch - p.bh)) >= unsigned(p.ew)
                                                      : false;
                    if (out) bits |= 1u << c;
                }
                uint32_t w[4];
#pragma unroll
                for (int cc = 0; cc < 4; ++cc)
                    w[cc] = (((bits >> (2 * cc)) & 1u) ? neg : 0u) |
                            (((bits >> (2 * cc + 1)) & 1u) ? (neg << 16) : 0u);
                *reinterpret_cast<uint4 *>(smem + C::kxv_off(v) + ptx::sw32_offset(r, half)) =
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
        if ((warp == C::W_LOAD || warp == C::W_LOAD1) && lane == 0) {
            // ============================================= TMA loaders, one
            // per stream: the box's queries, then K and V of each key tile in
            // the order the issuer consumes them.  The rings run on across
            // boxes: key tile g of the stream (counted over its boxes) goes to
            // K stage g % KS and V stage g % VS.
            const int tt = warp == C::W_LOAD ? 0 : 1;
            ptx::prefetch_tmap(&tq);
            ptx::prefetch_tmap(&tk);
            ptx::prefetch_tmap(&tv);
            const uint64_t pol_kv = ptx::l2_policy_evict_last();
            const uint64_t pol_q = ptx::l2_policy_evict_first();
            int G = 0;                        // key tiles of earlier boxes
            int q_issued = 0;                 // query loads issued
            bool ok = true;
            int ci = 0;
            for (int b = na_stream_box(p, tt, 0); ok && b >= 0; b = na_stream_box(p, tt, ++ci)) {
                const NaBox x = na_box(p, b, KT, KH);
                // the queries of box ci overwrite those of box ci - 1 once every
                // Q K^T that read them has completed.  q_free is one phase per
                // box, and its phase ci needs the queries loaded here, so it is
                // never two phases ahead of this wait.
                if (ci > 0 && !ptx::mbar_wait_or_abort(&bars->q_free[tt], (ci - 1) & 1, p.err, abort)) {
                    ok = false;
                    break;
                }
                // the box's first two K tiles count on its queries' barrier
                // (registered before its arrival), so that no step waits for
                // a copy of a later box
                const int nt = x.g.ntiles;
                ptx::mbar_expect_tx(&bars->q_full[tt], imin(nt, 2) * C::KV_BYTES);
                ptx::mbar_arrive_expect_tx(&bars->q_full[tt], rows * 128);
                ptx::tma_load_5d(smem + C::OFF_Q + tt * C::PANEL, &tq, 0, x.g.w0, x.g.h0, x.g.t0, x.bhd,
                                 &bars->q_full[tt], pol_q);
                q_issued = ci + 1;
                for (int j = 0; j < x.g.ntiles; ++j) {
                    const int g = G + j;
                    int kt_, kh_, kw_;
                    na_key_box(x.g, KT, KH, j, kt_, kh_, kw_);
                    // both stages of tile g are free once Q K^T (g - 2) has
                    // completed.  Q K^T (g) needs the copies issued here, so
                    // s_full is never two phases ahead of this wait.
                    if (g >= 2 && !ptx::mbar_wait_or_abort(&bars->s_full[2 * tt + (g & 1)], ((g - 2) >> 1) & 1,
                                                           p.err, abort)) {
                        ok = false;
                        break;
                    }
                    // K(g) serves step g - 2 (the box's first two: its queries'
                    // barrier), V(g) step g
                    uint64_t *bk = j >= 2 ? &bars->ready[tt][(g - 2) & 3] : &bars->q_full[tt];
                    if (j >= 2) ptx::mbar_arrive_expect_tx(bk, C::KV_BYTES);
                    ptx::tma_load_5d(smem + C::k_off(g % C::KS, tt), &tk, 0, kw_, kh_, kt_, x.bhd, bk, pol_kv);
                    uint64_t *bv = &bars->ready[tt][g & 3];
                    ptx::mbar_arrive_expect_tx(bv, C::KV_BYTES);
                    ptx::tma_load_5d(smem + C::v_off(g % C::VS, tt), &tv, 0, kw_, kh_, kt_, x.bhd, bv, pol_kv);
                }
                // the box's last two steps have no K tile two ahead in the box
                if (ok)
                    for (int j = imax(0, nt - 2); j < nt; ++j) ptx::mbar_arrive(&bars->ready[tt][(G + j) & 3]);
                G += nt;
            }
            // after a timeout elsewhere: let the copies this thread issued land
            // before the CTA's shared memory is released.  Their barriers also
            // wait for softmax arrivals that may never come, so wait for the
            // queries' barrier (bounded) and then a fixed 50 us, far above the
            // latency of a copy.
            if (*abort) {
                if (q_issued > 0) ptx::mbar_wait(&bars->q_full[tt], (q_issued - 1) & 1, nullptr);
                const unsigned long long t0 = global_timer_ns();
                while (global_timer_ns() - t0 < 50000ull) {
                }
            }
        } else if ((warp == C::W_MMA || warp == C::W_MMA1) && lane == 0) {
            // ============================================= MMA issuers: one
            // thread per stream (warps of different SM sub-partitions)
            const int tt = warp == C::W_MMA ? 0 : 1;
            const uint32_t id_qk = ptx::idesc_16_f32(kBM, kBN, false, F16);
            const uint32_t id_pv = ptx::idesc_16_f32(kBM, kD, true, F16);
            // descriptors are built once; a k-step, stage or tile only moves the
            // start-address field (byte address >> 4, no carry below 256 KB)
            constexpr uint32_t HI128 = ptx::desc_hi_sw128(1024), HI32 = ptx::desc_hi_sw32(256);
            const uint32_t dq = ptx::desc_lo_sw128(ptx::smem_addr(smem + C::OFF_Q + tt * C::PANEL), 16);
            const uint32_t dk0 = ptx::desc_lo_sw128(ptx::smem_addr(smem + C::k_off(0, tt)), 16);
            const uint32_t dv0 = ptx::desc_lo_sw128(ptx::smem_addr(smem + C::v_off(0, tt)), C::KV_BYTES);
            uint32_t dqx = 0, dkx0 = 0;
            if constexpr (PEN) {
                dqx = ptx::desc_lo_sw32(ptx::smem_addr(smem + C::qx_off(tt)));
                dkx0 = ptx::desc_lo_sw32(ptx::smem_addr(smem + C::kxv_off(0)));
            }
            int hq = 0, wq = 0, nhq = 1, nwq = 1;   // union h / w chunk of the next Q K^T (of nhq / nwq)
            // S(g) of the stream's key tile g into buffer g % 2
            auto issue_qk = [&](int g) {
                const uint32_t b0 = dk0 + uint32_t(((g % C::KS) * C::STAGE_BYTES) >> 4);
                const uint32_t d = tmem + C::tm_s(tt, g & 1);
#pragma unroll
                for (int kk = 0; kk < kD / 16; ++kk)
                    ptx::mma_ss(d, ptx::desc_join(dq + uint32_t(kk * 2), HI128),
                                ptx::desc_join(b0 + uint32_t(kk * 2), HI128), id_qk, kk > 0);
                if constexpr (PEN) {
                    // + window penalties: one more k-step over the 16 extra
                    // channels with the key tile's (h chunk, w chunk) tile
                    const uint32_t b = dkx0 + uint32_t(((hq * p.nwv + wq) * C::KX_BYTES) >> 4);
                    if (++wq == nwq) {
                        wq = 0;
                        if (++hq == nhq) hq = 0;
                    }
                    ptx::mma_ss(d, ptx::desc_join(dqx, HI32), ptx::desc_join(b, HI32), id_qk, 1u);
                }
                ptx::tc_commit(&bars->s_full[2 * tt + (g & 1)]);
            };
            // O (+)= P(g) V(g); the first key tile of a box overwrites O
            auto issue_pv = [&](int g, bool first) {
                const uint32_t b0 = dv0 + uint32_t(((g % C::VS) * C::STAGE_BYTES) >> 4);
                const uint32_t a0 = tmem + C::tm_s(tt, g & 1);
#pragma unroll
                for (int kk = 0; kk < kBN / 16; ++kk)
                    ptx::mma_ts(tmem + C::tm_o(tt), a0 + kk * 8,
                                ptx::desc_join(b0 + uint32_t(kk * (2048 >> 4)), HI128), id_pv,
                                (!first || kk > 0) ? 1u : 0u);
                ptx::tc_commit(&bars->o_done[2 * tt + (g & 1)]);
            };
            bool ok = true;
            int G = 0;                        // key tiles of the stream's earlier boxes
            // stream 1 starts once issuer 0 has issued p.stagger P V (or run out
            // of boxes): one arrival, one phase, waited for once
            bool go_sent = tt != 0;
            auto send_go = [&]() {
                if (!go_sent) ptx::mbar_arrive(&bars->go);
                go_sent = true;
            };
            if (p.stagger <= 0) send_go();
            if (tt != 0) ok = ptx::mbar_wait_or_abort(&bars->go, 0, p.err, abort);
            int ci = 0;
            for (int b = na_stream_box(p, tt, 0); ok && b >= 0; b = na_stream_box(p, tt, ++ci)) {
                const NaBox x = na_box(p, b, KT, KH);
                const int nt = x.g.ntiles;
                ok = ptx::mbar_wait_or_abort(&bars->q_full[tt], ci & 1, p.err, abort);
                if (!ok) break;
                if constexpr (PEN) {
                    // the softmax of this stream has written the box's query
                    // channels (after reading every S of the previous box)
                    ok = ptx::mbar_wait_or_abort(&bars->chan_ready[tt], ci & 1, p.err, abort);
                    if (!ok) break;
                    hq = wq = 0;
                    nhq = x.g.nhc;
                    nwq = x.g.nwc;
                }
                ptx::tc_fence_after();
                // Q K^T of key tile j; q_free right behind the box's last one
                auto next_qk = [&](int j) {
                    const int g = G + j;
                    if (!ok) return;
                    issue_qk(g);
                    if (j == nt - 1) ptx::tc_commit(&bars->q_free[tt]);
                };
                for (int j = 0; ok && j < 2 && j < nt; ++j) next_qk(j);
                for (int j = 0; ok && j < nt; ++j) {
                    const int g = G + j;
                    // P V (j) once the softmax has written P(j) and V(j) has landed,
                    // and K(j + 2) has landed for the Q K^T behind it
                    ok = ptx::mbar_wait_or_abort(&bars->ready[tt][g & 3], (g >> 2) & 1, p.err, abort);
                    if (!ok) break;
                    ptx::tc_fence_after();
                    issue_pv(g, j == 0);
                    // then Q K^T (j + 2) into the buffer P(j) came from
                    if (j + 2 < nt) next_qk(j + 2);
                    if (!ok) break;
                    if (g + 1 >= p.stagger) send_go();
                }
                G += nt;
            }
            send_go();
            // drain: every MMA of both issuers has completed before TMEM is freed
            ptx::tc_commit(&bars->drain);
            ptx::mbar_wait(&bars->drain, 0, p.err);
        }
    } else {
        // ================================================= softmax warpgroups
        ptx::regs_increase<C::REGS_SOFTMAX>();
        const int t = warp >> 2;                 // stream
        const int quarter = warp & 3;            // TMEM lanes [32 quarter, 32 quarter + 32)
        const int row = quarter * 32 + lane;     // query row within the box
        const uint32_t lane_base = tmem + (uint32_t(quarter * 32) << 16);
        const uint32_t o_addr = lane_base + C::tm_o(t);
        const float cl = p.c_log2;
        constexpr int NG = kBN / 16;             // 16-key groups per key tile
        const int dt = row / (p.bh * p.bw), dh = (row / p.bw) % p.bh, dw = row % p.bw;

        // waits for P V (gg) of this stream (and every earlier one: one
        // thread's MMAs complete in issue order).  Valid once P V (gg - 2) is known
        // complete: it is while the softmax holds S(gg), issued after it.
        auto wait_pv = [&](int gg) -> bool {
            if (!__all_sync(0xffffffffu, ptx::mbar_wait_or_abort(&bars->o_done[2 * t + (gg & 1)],
                                                                 (gg >> 1) & 1, p.err, abort)))
                return false;
            ptx::tc_fence_after();
            return true;
        };

        bool ok = true;
        int G = 0;                               // key tiles of the stream's earlier boxes
        // This row's query channels for box gx: one-hot at the offsets of
        // its h and w windows from the union origin (zero for a row outside
        // the box or the grid).  Every Q K^T of the previous box must have
        // completed (this warpgroup has read all their scores); the issuer
        // waits for chan_ready before the box's first one.
        auto write_qx = [&](const NaTile &gx) {
            const int qh = gx.h0 + dh, qw = gx.w0 + dw;
            const bool in = row < rows && gx.t0 + dt < p.T && qh < p.Hg && qw < p.W;
            const int ch0 = in ? na_window_start(qh, p.Hg, p.kh) - gx.u0h : -1;
            const int ch1 = in ? p.bh + na_window_start(qw, p.W, p.kw) - gx.u0w : -1;
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                uint32_t w[4] = {0u, 0u, 0u, 0u};
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const int c = half * 8 + e;
                    if (c == ch0 || c == ch1) w[e >> 1] |= uint32_t(H16<F16>::kOne) << ((e & 1) * 16);
                }
                *reinterpret_cast<uint4 *>(smem + C::qx_off(t) + ptx::sw32_offset(row, half)) =
                    make_uint4(w[0], w[1], w[2], w[3]);
            }
            ptx::fence_proxy_async_smem();
            ptx::mbar_arrive(&bars->chan_ready[t]);
        };
        int ci = 0;
        int b = na_stream_box(p, t, 0);          // the stream's box ci
        if constexpr (PEN) {
            if (b >= 0) write_qx(na_box(p, b, KT, KH).g);
        }
        while (ok && b >= 0) {
            const NaBox x = na_box(p, b, KT, KH);
            const int nt = x.g.ntiles;
            const NaTile &gt = x.g;

            // query of this row and its window
            const int qt = gt.t0 + dt, qh = gt.h0 + dh, qw = gt.w0 + dw;
            const bool qvalid = row < rows && qt < p.T && qh < p.Hg && qw < p.W;
            const int wst = na_window_start(imin(qt, p.T - 1), p.T, p.kt);
            int wsh = 0, wsw = 0;
            if constexpr (!PEN) {
                wsh = na_window_start(imin(qh, p.Hg - 1), p.Hg, p.kh);
                wsw = na_window_start(imin(qw, p.W - 1), p.W, p.kw);
            }

            float m = -INFINITY, l = 0.f;
            int tc = 0, hc = 0, wc = 0;          // key sub-box counters (w fastest, then h, then t)
            // t window per 16-key group of the current t chunk (group gq holds
            // frame kt0 + gq / KH): bit gq of gmask clear -> P = 0 there; wlive:
            // the groups any row of the warp sees.  Both change with tc only.
            auto group_mask = [&](int tcc) -> uint32_t {
                uint32_t gmv = 0u;
                if (qvalid) {
                    const int kt0 = gt.u0t + tcc * KT;
#pragma unroll
                    for (int gq = 0; gq < NG; ++gq)
                        if (unsigned(kt0 + gq / KH - wst) < unsigned(p.et)) gmv |= 1u << gq;
                }
                return gmv;
            };
            uint32_t gmask = group_mask(0);
            uint32_t wlive = __reduce_or_sync(0xffffffffu, gmask);
            for (int j = 0; j < nt; ++j) {
                const int gg = G + j;
                const uint32_t s_addr = lane_base + C::tm_s(t, gg & 1);
                if (!__all_sync(0xffffffffu, ptx::mbar_wait_or_abort(&bars->s_full[2 * t + (gg & 1)],
                                                                     (gg >> 1) & 1, p.err, abort))) {
                    ok = false;
                    break;
                }
                ptx::tc_fence_after();

                const int kh0 = gt.u0h + hc * KH, kw0 = gt.u0w + wc * kKW;
                bool new_tc = false;
                if (++wc == gt.nwc) {
                    wc = 0;
                    if (++hc == gt.nhc) {
                        hc = 0;
                        ++tc;
                        new_tc = true;
                    }
                }

                float sv[kBN];
#pragma unroll
                for (int c = 0; c < kBN / 32; ++c)
                    ptx::tmem_ld32(s_addr + c * 32, *reinterpret_cast<uint32_t(*)[32]>(&sv[c * 32]));
                ptx::tmem_wait_ld();

                if constexpr (!PEN) {
                    // f16: the h and w window tests per key.  Key e of the (KT, KH, 16)
                    // sub-box sits at h = kh0 + (e / 16) % KH, w = kw0 + e % 16; wm / hm
                    // hold the in-window w columns / h rows of this row.
                    const int lw = wsw - kw0, lh = wsh - kh0;
                    const int aw = imax(lw, 0), bw = imin(lw + p.ew, kKW);
                    const int ah = imax(lh, 0), bh_ = imin(lh + p.eh, KH);
                    const uint32_t wm = aw < bw ? ((1u << bw) - 1u) & ~((1u << aw) - 1u) : 0u;
                    const uint32_t hm = ah < bh_ ? ((1u << bh_) - 1u) & ~((1u << ah) - 1u) : 0u;
#pragma unroll
                    for (int gq = 0; gq < NG; ++gq) {
                        const bool hin = (hm >> (gq % KH)) & 1u;
#pragma unroll
                        for (int i = 0; i < 16; ++i)
                            if (!hin || !((wm >> i) & 1u)) sv[gq * 16 + i] = -INFINITY;
                    }
                }

                // 32-key chunks that no row of this warp may see: P = 0 without
                // exponentials
                // (gmask and wlive of this key tile; the next t chunk's below)

                // P = 2^(x - m) in 16-bit over S (groups outside gm: P = 0);
                // returns the tile's row sum (fp32)
                auto emit_p = [&](float nmu, uint32_t gm) -> float {
                    float acc[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i) acc[i] = 0.f;
#pragma unroll
                    for (int c = 0; c < kBN / 32; ++c) {
                        uint32_t pk[16];
                        if (((wlive >> (2 * c)) & 3u) == 0u) {
#pragma unroll
                            for (int e = 0; e < 16; ++e) pk[e] = 0u;
                            ptx::tmem_st16(s_addr + c * 16, pk);
                            continue;
                        }
                        const float n0 = ((gm >> (2 * c)) & 1u) ? nmu : -INFINITY;
                        const float n1 = ((gm >> (2 * c + 1)) & 1u) ? nmu : -INFINITY;
#pragma unroll
                        for (int e = 0; e < 16; ++e) {
                            const float nm = e < 8 ? n0 : n1;
                            float x0, x1;
                            ptx::ffma2(x0, x1, sv[c * 32 + 2 * e], sv[c * 32 + 2 * e + 1], cl, cl, nm, nm);
                            const float p0 = ptx::ex2(x0), p1 = ptx::ex2(x1);
                            ptx::fadd2(acc[(2 * e) & 7], acc[(2 * e + 1) & 7], acc[(2 * e) & 7],
                                       acc[(2 * e + 1) & 7], p0, p1);
                            pk[e] = H16<F16>::pack(p0, p1);
                        }
                        ptx::tmem_st16(s_addr + c * 16, pk);
                    }
                    return ((acc[0] + acc[1]) + (acc[2] + acc[3])) + ((acc[4] + acc[5]) + (acc[6] + acc[7]));
                };

                // ---- fast path: exponentiate against m as it stands.  P only
                //      has to stay finite in its 16-bit type: a tile whose row sum
                //      exceeds 2^24 (2^15 for f16, largest finite 65504) or is not
                //      finite (scores far above m, or m still the garbage of a row
                //      whose first tiles were all outside its window) is redone
                //      against its own maximum.
                bool fast = j > 0 && __all_sync(0xffffffffu, !(gmask != 0u && m == -INFINITY));
                if (fast) {
                    const float lt = emit_p(-m, gmask);
                    if (__any_sync(0xffffffffu, !(lt <= (F16 ? 32768.f : 16777216.f))))
                        fast = false;             // redo the tile (P is rewritten below)
                    else
                        l += lt;
                }
                if (!fast) {
                    // ---- tile maximum over the groups this row may see
                    float tmax = -INFINITY;
#pragma unroll
                    for (int gq = 0; gq < NG; ++gq) {
                        float mx[8];
#pragma unroll
                        for (int i = 0; i < 8; ++i) mx[i] = fmaxf(sv[gq * 16 + i], sv[gq * 16 + 8 + i]);
                        const float gmx = ptx::fmax3(ptx::fmax3(mx[0], mx[1], mx[2]),
                                                     ptx::fmax3(mx[3], mx[4], mx[5]), fmaxf(mx[6], mx[7]));
                        if ((gmask >> gq) & 1u) tmax = fmaxf(tmax, gmx);
                    }
                    const float mt = tmax * cl;  // cl > 0: max commutes with the scaling
                    // ---- rows whose max moves: a row whose max grows by more
                    //      than 8, or that sees its window for the first time (m
                    //      = -inf, as every row on the box's first key tile).  Only
                    //      the first kind holds anything to rescale (a row at m =
                    //      -inf has had P = 0 so far: O and l are 0), and only
                    //      then must the previous P V be done first.
                    const bool want = mt > m + 8.f;
                    const bool resc = want && m != -INFINITY;
                    const bool any_resc = __any_sync(0xffffffffu, resc);
                    if (any_resc && !wait_pv(gg - 1)) {
                        ok = false;
                        break;
                    }
                    if (any_resc) {
                        // rows that move a finite m scale their O row; the others multiply by 1
                        const float f = resc ? ptx::ex2(m - mt) : 1.f;
#pragma unroll
                        for (int c = 0; c < kD / 32; ++c) {
                            uint32_t ov[32];
                            ptx::tmem_ld32(o_addr + c * 32, ov);
                            ptx::tmem_wait_ld();
#pragma unroll
                            for (int e = 0; e < 32; e += 2) {
                                float a0, a1;
                                ptx::ffma2(a0, a1, __uint_as_float(ov[e]), __uint_as_float(ov[e + 1]), f, f,
                                           0.f, 0.f);
                                ov[e] = __float_as_uint(a0);
                                ov[e + 1] = __float_as_uint(a1);
                            }
                            ptx::tmem_st32(o_addr + c * 32, ov);
                        }
                        l *= f;
                    }
                    if (want) m = mt;
                    l += emit_p((m == -INFINITY) ? 0.f : -m, gmask);
                }
                ptx::tmem_wait_st();
                ptx::tc_fence_before();
                ptx::mbar_arrive(&bars->ready[t][gg & 3]);
                if (new_tc) {
                    gmask = group_mask(tc);
                    wlive = __reduce_or_sync(0xffffffffu, gmask);
                }
            }
            if (!ok) break;

            // ---- the next box's query channels before this box's outputs:
            //      every Q K^T of the stream has completed (its last scores
            //      are read), so the issuer can start the next box's Q K^T
            //      while the outputs are written
            const int nb = na_stream_box(p, t, ci + 1);
            if constexpr (PEN) {
                if (nb >= 0) write_qx(na_box(p, nb, KT, KH).g);
            }

            // ---- epilogue: O / l -> 16-bit -> global.  The issuer overwrites O
            //      with the next box's first P V only after this warpgroup has
            //      written that box's P(0), i.e. after these reads.
            if (!wait_pv(G + nt - 1)) {
                ok = false;
                break;
            }
            const float inv = 1.f / l;
            typename H16<F16>::T *orow = nullptr;
            if (qvalid)
                orow = static_cast<typename H16<F16>::T *>(p.o) +
                       ((size_t(x.bhd) * (size_t(p.T) * p.Hg * p.W)) + (size_t(qt) * p.Hg + qh) * p.W + qw) * kD;
#pragma unroll
            for (int c = 0; c < kD / 32; ++c) {
                uint32_t ov[32];
                ptx::tmem_ld32(o_addr + c * 32, ov);
                ptx::tmem_wait_ld();
                if (qvalid) {
                    uint4 w4[4];
                    uint32_t *wp = reinterpret_cast<uint32_t *>(w4);
#pragma unroll
                    for (int e = 0; e < 16; ++e)
                        wp[e] = H16<F16>::pack(__uint_as_float(ov[2 * e]) * inv, __uint_as_float(ov[2 * e + 1]) * inv);
                    // streaming stores: the outputs are not read again here, and
                    // evicting them early keeps the key tiles in L2 and leaves
                    // less to write back after the kernel
                    uint4 *dst = reinterpret_cast<uint4 *>(orow + c * 32);
#pragma unroll
                    for (int e = 0; e < 4; ++e) __stcs(dst + e, w4[e]);
                }
            }
            G += nt;
            b = nb;
            ++ci;
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

// ------------------------------------------------------------- host side

// Query box and key sub-box: at most 128 queries per box and key tiles of KT
// frames x KH rows x 16 columns (KT KH = 6, 96 keys), minimising the key tiles
// -- i.e. the (query row, key) slots the MMAs compute -- over all boxes.
bool plan_na(int T, int Hg, int W, const int kern[3], int &bt, int &bh, int &bw, int &KT, int &KH,
             double &tiles) {
    const int ext[3] = {T, Hg, W};
    constexpr int kShapes[4][2] = {{1, 6}, {2, 3}, {3, 2}, {6, 1}};
    double best = -1;
    for (int cbt = 1; cbt <= imin(T, 128); ++cbt)
        for (int cbh = 1; cbh <= imin(Hg, 128 / cbt); ++cbh)
            for (int cbw = 1; cbw <= imin(W, 128 / (cbt * cbh)); ++cbw) {
                if (cbt * cbh * cbw < imin(64, T * Hg * W)) continue;   // keep MMA rows busy
                if (cbh + cbw > 16) continue;                // h and w offsets fit 16 channels
                for (const auto &sh : kShapes) {
                    const int ckt = sh[0], ckh = sh[1];
                    // distinct key penalty tiles of a box (h chunks x w chunks) must fit
                    const int nh_max = cdiv(imin(cbh + imin(kern[1], Hg) - 1, Hg), ckh);
                    const int nw_max = cdiv(imin(cbw + imin(kern[2], W) - 1, W), kKW);
                    if (nh_max * nw_max > kMaxPenaltyTiles) continue;
                    // key tiles over all boxes = sum_t(t chunks) * sum_h(h chunks) * sum_w(w chunks)
                    const int b[3] = {cbt, cbh, cbw}, chunk[3] = {ckt, ckh, kKW};
                    double axis[3];
                    for (int a = 0; a < 3; ++a) {
                        const int keff = imin(kern[a], ext[a]);
                        double acc = 0;
                        for (int i0 = 0; i0 < ext[a]; i0 += b[a]) {
                            const int i1 = imin(i0 + b[a], ext[a]) - 1;
                            const int u = na_window_start(i1, ext[a], kern[a]) + keff -
                                          na_window_start(i0, ext[a], kern[a]);
                            acc += cdiv(u, chunk[a]);
                        }
                        axis[a] = acc;
                    }
                    const double cost = axis[0] * axis[1] * axis[2];
                    if (best < 0 || cost < best) {
                        best = cost;
                        bt = cbt; bh = cbh; bw = cbw; KT = ckt; KH = ckh;
                        tiles = cost;
                    }
                }
            }
    return best > 0;
}

// Plans are cached per (grid, kernel): the search is a few thousand candidates.
struct NaPlan {
    int bt, bh, bw, KT, KH;
    double tiles;            // key tiles of all boxes of one (batch, head)
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
    pl.ok = plan_na(T, Hg, W, kern, pl.bt, pl.bh, pl.bw, pl.KT, pl.KH, pl.tiles);
    Entry &e = cache[used < 64 ? used++ : 63];
    for (int a = 0; a < 6; ++a) e.key[a] = key[a];
    e.plan = pl;
    return pl;
}

template <int KSH, bool F16 = false>
attn_status_t launch_na(const Ctx &c, const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                        const NaParams &p) {
    using C = NaCfg<!F16>;
    static int done_mask = 0;
    static int regs = -1;
    auto kern = tc_na_kernel<KSH, F16>;
    if (!ensure_smem_attr(reinterpret_cast<const void *>(kern), C::SMEM, c.device, &done_mask))
        return ATTN_ERR_RESOURCE;
    // the warpgroups re-split the launch's register file with setmaxnreg; the
    // split is only valid for the per-thread count it was computed for
    if (regs < 0) {
        cudaFuncAttributes fa;
        if (cudaFuncGetAttributes(&fa, reinterpret_cast<const void *>(kern)) != cudaSuccess) {
            cudaGetLastError();
            return ATTN_ERR_CUDA;
        }
        regs = fa.numRegs;
    }
    if (regs != C::REGS_LAUNCH) return ATTN_ERR_UNSUPPORTED;
    // one CTA per SM (the shared memory allows no second), each running two
    // streams of boxes
    const int grid = imin(cdiv(p.n_boxes, kNQ), imax(1, c.sm_count));
    kern<<<grid, C::NT, C::SMEM, c.stream>>>(tq, tk, tv, p);
    return launch_status(kFamTcNa);
}

}  // namespace

bool tc_na3d_supported(int B, int H, int T, int Hg, int W, int D, const int kernel[3]) {
    return D == kD && tma_encode_available() && cached_plan(T, Hg, W, kernel).ok;
}

attn_status_t tc_na3d(const Ctx &c, attn_dtype_t dt, const void *q, const void *k, const void *v,
                      void *o, int B, int H, int T, int Hg, int W, int D, const int kernel[3],
                      float scale) {
    const bool f16 = dt == ATTN_F16;
    const NaPlan pl = cached_plan(T, Hg, W, kernel);
    if (!pl.ok || D != kD) return ATTN_ERR_UNSUPPORTED;
    NaParams p{};
    p.bt = pl.bt; p.bh = pl.bh; p.bw = pl.bw; p.KT = pl.KT; p.KH = pl.KH;
    CUtensorMap tq, tk, tv;
    const uint64_t dims[5] = {uint64_t(D), uint64_t(W), uint64_t(Hg), uint64_t(T), uint64_t(B) * H};
    const uint32_t qbox[5] = {64, uint32_t(p.bw), uint32_t(p.bh), uint32_t(p.bt), 1};
    const uint32_t kbox[5] = {64, uint32_t(kKW), uint32_t(p.KH), uint32_t(p.KT), 1};
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
    p.nbt = cdiv(T, p.bt);
    p.nbh = cdiv(Hg, p.bh);
    p.nbw = cdiv(W, p.bw);
    p.nhv = cdiv(imin(p.bh + p.eh - 1, Hg), p.KH);   // the planner keeps nhv nwv <= 7
    p.nwv = cdiv(imin(p.bw + p.ew - 1, W), kKW);
    const long long boxes = (long long)p.nbt * p.nbh * p.nbw * B * H;
    if (boxes > 0x7fffffffLL - 4096) return ATTN_ERR_UNSUPPORTED;   // box indices + 2 grid fit int
    p.n_boxes = int(boxes);
    // stream 1 starts half a mean box (in key tiles) behind stream 0
    p.stagger = int(0.5 * pl.tiles / (double(p.nbt) * p.nbh * p.nbw) + 0.5);
    // the planner's key sub-box shapes have compile-time kernels (bf16)
    if (f16) return launch_na<0, true>(c, tq, tk, tv, p);
    switch (p.KT * 10 + p.KH) {
        case 16: return launch_na<16>(c, tq, tk, tv, p);
        case 23: return launch_na<23>(c, tq, tk, tv, p);
        case 32: return launch_na<32>(c, tq, tk, tv, p);
        default: return launch_na<0>(c, tq, tk, tv, p);
    }
}

}  // namespace attn
