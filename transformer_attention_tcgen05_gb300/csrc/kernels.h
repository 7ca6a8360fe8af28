// Host-side launchers of libattn's kernels (internal; the public ABI is include/libattn.h).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "libattn.h"

namespace attn {

struct Ctx {
    cudaStream_t stream;
    unsigned *err;      // device error word of the current device
    int device;
    int sm_count;
};

enum KernelFamily : int {
    kFamSimt = 0,
    kFamTcFlash = 1,
    kFamDecode = 2,
    kFamRope = 3,
    kFamNaStarts = 4,
    kFamTcNa = 5,
    kFamKvAppend = 6,
    kFamDebug = 7,
    kFamCount = 8,
};

void count_launch(int family);

// The per-device context (stream, device error word, SM count) of a call.
attn_status_t context_for(void *stream, Ctx *c);

// Converts the result of a launch into a status (and counts it on success).
attn_status_t launch_status(int family);

// Sets the dynamic shared-memory limit of `func` once per device.
bool ensure_smem_attr(const void *func, size_t bytes, int device, int *done_mask);

// 16-bit (bf16 or f16) TMA tensor map with 128-byte swizzle; dims and box
// innermost first (dims[0] = D), the tensor packed.  False if the driver's
// encoder is unavailable or rejects the map.
bool make_tmap(CUtensorMap *m, const void *base, int rank, const uint64_t *dims, const uint32_t *box,
               bool f16 = false);
bool tma_encode_available();

// Element strides of a [B, heads, N, D] tensor with D contiguous.
struct TensorStrides {
    long long b, h, n;
};

// fp32 / generic SIMT flash attention (exact FFMA for fp32 storage).
attn_status_t simt_full(const Ctx &c, attn_dtype_t dt, const void *q, const void *k,
                        const void *v, void *o, int B, int H, int Nq, int Nkv, int D,
                        float scale, const TensorStrides *st = nullptr);
attn_status_t simt_na3d(const Ctx &c, attn_dtype_t dt, const void *q, const void *k,
                        const void *v, void *o, int B, int H, int T, int Hg, int W, int D,
                        const int kernel[3], float scale, const TensorStrides *st = nullptr);
attn_status_t na_starts(const Ctx &c, int T, int Hg, int W, const int kernel[3],
                        int32_t *starts);

// RoPE prologue: rotated copies of q and k into qr / kr (same dtype).
attn_status_t rope_rotate_qk(const Ctx &c, attn_dtype_t dt, const void *q, const void *k,
                             void *qr, void *kr, int BH, int N, int D, const int32_t *pos,
                             const int axes_dim[4], float theta);

// KV-cache append at the device-side position seq_len[b] (optionally advancing it);
// ring: the cache keeps the last Lmax tokens, token t in row t % Lmax.
attn_status_t kv_append(const Ctx &c, attn_dtype_t dt, void *kc, void *vc, const void *kn,
                        const void *vn, int32_t *seq_len, int B, int Hkv, int Lmax, int D,
                        int advance, bool ring = false);

// Split-KV GQA decode (bf16 or f16 cache).
size_t decode_workspace_bytes(int B, int Hq, int Hkv, int Lmax, int D);
attn_status_t decode_gqa(const Ctx &c, attn_dtype_t dt, const void *q, const void *k,
                         const void *v, const int32_t *seq_len, void *o, int B, int Hq, int Hkv,
                         int Lmax, int D, float scale, void *ws, size_t ws_bytes,
                         bool ring = false);

// tcgen05 (tensor-core) flash attention, bf16 or f16: full and neighborhood.
// st: strides of q, k, v, o (nullptr: contiguous).
attn_status_t tc_full(const Ctx &c, attn_dtype_t dt, const void *q, const void *k, const void *v,
                      void *o, int B, int H, int Nq, int Nkv, int D, float scale,
                      const TensorStrides *st = nullptr);
bool tc_full_supported(int B, int H, int Nq, int Nkv, int D);
attn_status_t tc_causal_gqa(const Ctx &c, attn_dtype_t dt, const void *q, const void *k,
                            const void *v, void *o, int B, int Hq, int Hkv, int N, int D,
                            float scale, const TensorStrides *st = nullptr);
attn_status_t simt_causal_gqa(const Ctx &c, attn_dtype_t dt, const void *q, const void *k,
                              const void *v, void *o, int B, int Hq, int Hkv, int N, int D,
                              float scale, const TensorStrides *st = nullptr);
attn_status_t tc_na3d(const Ctx &c, attn_dtype_t dt, const void *q, const void *k, const void *v,
                      void *o, int B, int H, int T, int Hg, int W, int D, const int kernel[3],
                      float scale);
bool tc_na3d_supported(int B, int H, int T, int Hg, int W, int D, const int kernel[3]);
// One 128 x 128 tile through both tcgen05 MMA forms (testing).
attn_status_t tc_selftest(const Ctx &c, const void *q, const void *k, const void *v,
                          const void *P, float *S, float *O, int D);

}  // namespace attn
