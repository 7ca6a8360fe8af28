// The C ABI of libattn (include/libattn.h): argument validation, per-device
// context, dispatch to the kernels, error reporting and launch counters.
#include <atomic>
#include <math.h>
#include <mutex>
#include <stdint.h>

#include "common.cuh"
#include "kernels.h"
#include "ptx.cuh"

namespace attn {

// Device error word: bounded waits and device-side checks raise it.
__device__ unsigned g_device_error = 0;

namespace {

constexpr int kMaxDevices = 64;
std::atomic<uint64_t> g_launches[kFamCount];

struct DevInfo {
    unsigned *err = nullptr;
    int sm_count = 0;
    bool ready = false;
};
DevInfo g_dev[kMaxDevices];
std::mutex g_dev_mutex;

attn_status_t get_ctx(void *stream, Ctx *c) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return ATTN_ERR_CUDA;
    }
    DevInfo &d = g_dev[dev];
    if (!d.ready) {
        std::lock_guard<std::mutex> lock(g_dev_mutex);
        if (!d.ready) {
            void *ptr = nullptr;
            int sms = 0;
            if (cudaGetSymbolAddress(&ptr, g_device_error) != cudaSuccess ||
                cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
                cudaGetLastError();
                return ATTN_ERR_CUDA;
            }
            d.err = static_cast<unsigned *>(ptr);
            d.sm_count = sms;
            d.ready = true;
        }
    }
    c->stream = static_cast<cudaStream_t>(stream);
    c->err = d.err;
    c->device = dev;
    c->sm_count = d.sm_count;
    return ATTN_OK;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

float resolve_scale(float scale, int D) {
    return (scale > 0.f && isfinite(scale)) ? scale : 1.0f / sqrtf(float(D));
}

bool valid_d(int D) { return D == 32 || D == 64 || D == 128; }

bool valid_dtype(attn_dtype_t dt) { return dt == ATTN_F32 || dt == ATTN_BF16 || dt == ATTN_F16; }

// bf16 and f16 run on the tensor cores where the shapes allow.
bool half_dtype(attn_dtype_t dt) { return dt == ATTN_BF16 || dt == ATTN_F16; }

size_t elem_size(attn_dtype_t dt) { return dt == ATTN_F32 ? 4 : 2; }

// A (batch, head or row) stride of a strided view: positive, a multiple of 16
// bytes and below 2^40 bytes (the tensor-memory-access unit's stride limits).
bool stride_ok(long long s, attn_dtype_t dt) {
    const long long bytes = s * (long long)elem_size(dt);
    return s >= 1 && s < (1ll << 38) && bytes % 16 == 0 && bytes < (1ll << 40);
}

// Extents whose element counts must stay below 2^31 per (batch, head) slice so
// that 32-bit row indices inside the kernels cannot overflow.
bool small_enough(long long rows, int D) { return rows > 0 && rows * D < (1ll << 31); }

// One thread waits on a shared-memory barrier that nothing ever completes:
// the bounded wait runs out after limit_ns, raises kDevTimeout and returns.
__global__ void wait_test_kernel(unsigned long long limit_ns, unsigned *err) {
    __shared__ uint64_t bar;
    ptx::mbar_init(&bar, 1);
    ptx::fence_barrier_init();
    ptx::mbar_wait_limit(&bar, 0, err, limit_ns);
}

}  // namespace

attn_status_t context_for(void *stream, Ctx *c) { return get_ctx(stream, c); }

void count_launch(int family) {
    if (family >= 0 && family < kFamCount) g_launches[family].fetch_add(1);
}

attn_status_t launch_status(int family) {
    if (cudaGetLastError() != cudaSuccess) return ATTN_ERR_CUDA;
    count_launch(family);
    return ATTN_OK;
}

bool ensure_smem_attr(const void *func, size_t bytes, int device, int *done_mask) {
    // done_mask is a per-kernel bitmask of devices already configured (device < 32).
    if (device < 32 && (__atomic_load_n(done_mask, __ATOMIC_ACQUIRE) & (1 << device))) return true;
    if (cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, int(bytes)) !=
        cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    if (device < 32) __atomic_fetch_or(done_mask, 1 << device, __ATOMIC_ACQ_REL);
    return true;
}

}  // namespace attn

using namespace attn;

extern "C" {

const char *attn_status_string(attn_status_t s) {
    switch (s) {
        case ATTN_OK: return "ok";
        case ATTN_ERR_INVALID_ARG: return "invalid argument";
        case ATTN_ERR_UNSUPPORTED: return "unsupported configuration";
        case ATTN_ERR_RESOURCE: return "insufficient resources (shared memory or workspace)";
        case ATTN_ERR_CUDA: return "CUDA error";
        case ATTN_ERR_TIMEOUT: return "bounded device wait timed out";
        case ATTN_ERR_DEVICE_CHECK: return "device-side check failed";
    }
    return "unknown status";
}

const char *attn_version(void) { return "libattn 0.1 sm_103a"; }

uint64_t attn_launch_count(int family) {
    if (family < 0 || family >= kFamCount) return 0;
    return g_launches[family].load();
}

attn_status_t attn_device_status(void *stream) {
    Ctx c;
    attn_status_t st = get_ctx(stream, &c);
    if (st != ATTN_OK) return st;
    if (cudaStreamSynchronize(c.stream) != cudaSuccess) {
        cudaGetLastError();
        return ATTN_ERR_CUDA;
    }
    unsigned word = 0;
    if (cudaMemcpy(&word, c.err, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess) {
        cudaGetLastError();
        return ATTN_ERR_CUDA;
    }
    if (word != 0) {
        const unsigned zero = 0;
        if (cudaMemcpy(c.err, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess) {
            cudaGetLastError();
            return ATTN_ERR_CUDA;
        }
    }
    if (word == kDevTimeout) return ATTN_ERR_TIMEOUT;
    if (word == kDevCheck) return ATTN_ERR_DEVICE_CHECK;
    return ATTN_OK;
}

attn_status_t attn_full_fwd(const void *q, const void *k, const void *v, void *o, int B, int H,
                            int Nq, int Nkv, int D, attn_dtype_t dtype, float scale,
                            void *stream) {
    if (!q || !k || !v || !o) return ATTN_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o))
        return ATTN_ERR_INVALID_ARG;
    if (B < 1 || H < 1 || Nq < 1 || Nkv < 1 || !valid_d(D) || !valid_dtype(dtype))
        return ATTN_ERR_INVALID_ARG;
    if (!small_enough(Nq, D) || !small_enough(Nkv, D) || (long long)B * H > 65535)
        return ATTN_ERR_UNSUPPORTED;
    if (o == q || o == k || o == v) return ATTN_ERR_INVALID_ARG;
    Ctx c;
    attn_status_t st = get_ctx(stream, &c);
    if (st != ATTN_OK) return st;
    const float sc = resolve_scale(scale, D);
    if (half_dtype(dtype) && tc_full_supported(B, H, Nq, Nkv, D)) {
        // a layout the tensor-map encoder refuses falls through to the SIMT kernel
        st = tc_full(c, dtype, q, k, v, o, B, H, Nq, Nkv, D, sc);
        if (st != ATTN_ERR_UNSUPPORTED) return st;
    }
    return simt_full(c, dtype, q, k, v, o, B, H, Nq, Nkv, D, sc);
}

// Strides of the four tensors of a strided call: q (B, Hq, Nq), k and v
// (B, Hkv, Nkv), o (B, Hq, Nq), each D-contiguous.  An extent-1 axis is never
// stepped along, so its stride is replaced by a valid one; the output's rows
// must be pairwise disjoint (sorted by stride, each axis' stride covers the
// span of the axes below it, the innermost span being the D-element row).
static attn_status_t parse_strides(const int64_t *const in[4], int B, int Hq, int Hkv, int Nq,
                                   int Nkv, int D, attn_dtype_t dtype, TensorStrides st[4]) {
    for (int i = 0; i < 4; ++i) {
        if (!in[i]) return ATTN_ERR_INVALID_ARG;
        const bool qo = i == 0 || i == 3;
        const long long ext[3] = {B, qo ? Hq : Hkv, qo ? Nq : Nkv};
        long long s[3];
        for (int a = 0; a < 3; ++a) {
            s[a] = ext[a] == 1 ? D : (long long)in[i][a];
            if (!stride_ok(s[a], dtype)) return ATTN_ERR_INVALID_ARG;
        }
        st[i] = TensorStrides{s[0], s[1], s[2]};
    }
    const long long ext[3] = {B, Hq, Nq};
    const long long s[3] = {st[3].b, st[3].h, st[3].n};
    int ord[3] = {0, 1, 2};
    for (int a = 0; a < 3; ++a)
        for (int b = a + 1; b < 3; ++b)
            if (s[ord[b]] < s[ord[a]]) { const int t = ord[a]; ord[a] = ord[b]; ord[b] = t; }
    long long span = D;
    for (int a = 0; a < 3; ++a) {
        if (ext[ord[a]] == 1) continue;
        if (s[ord[a]] < span) return ATTN_ERR_INVALID_ARG;
        span = s[ord[a]] * ext[ord[a]];
    }
    return ATTN_OK;
}

attn_status_t attn_full_fwd_strided(const void *q, const void *k, const void *v, void *o,
                                    int B, int H, int Nq, int Nkv, int D,
                                    const int64_t q_strides[3], const int64_t k_strides[3],
                                    const int64_t v_strides[3], const int64_t o_strides[3],
                                    attn_dtype_t dtype, float scale, void *stream) {
    if (!q || !k || !v || !o) return ATTN_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o))
        return ATTN_ERR_INVALID_ARG;
    if (B < 1 || H < 1 || Nq < 1 || Nkv < 1 || !valid_d(D) || !valid_dtype(dtype))
        return ATTN_ERR_INVALID_ARG;
    if ((long long)B * H > 65535) return ATTN_ERR_UNSUPPORTED;
    if (o == q || o == k || o == v) return ATTN_ERR_INVALID_ARG;
    const int64_t *const in[4] = {q_strides, k_strides, v_strides, o_strides};
    TensorStrides st[4];
    attn_status_t status = parse_strides(in, B, H, H, Nq, Nkv, D, dtype, st);
    if (status != ATTN_OK) return status;
    Ctx c;
    status = get_ctx(stream, &c);
    if (status != ATTN_OK) return status;
    const float sc = resolve_scale(scale, D);
    if (half_dtype(dtype) && tc_full_supported(B, H, Nq, Nkv, D)) {
        status = tc_full(c, dtype, q, k, v, o, B, H, Nq, Nkv, D, sc, st);
        if (status != ATTN_ERR_UNSUPPORTED) return status;
    }
    return simt_full(c, dtype, q, k, v, o, B, H, Nq, Nkv, D, sc, st);
}

attn_status_t attn_causal_gqa_fwd_strided(const void *q, const void *k, const void *v, void *o,
                                          int B, int Hq, int Hkv, int N, int D,
                                          const int64_t q_strides[3], const int64_t k_strides[3],
                                          const int64_t v_strides[3], const int64_t o_strides[3],
                                          attn_dtype_t dtype, float scale, void *stream) {
    if (!q || !k || !v || !o) return ATTN_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o))
        return ATTN_ERR_INVALID_ARG;
    if (B < 1 || Hq < 1 || Hkv < 1 || N < 1 || Hq % Hkv != 0 || !valid_d(D) || !valid_dtype(dtype))
        return ATTN_ERR_INVALID_ARG;
    if ((long long)B * Hq > 65535) return ATTN_ERR_UNSUPPORTED;
    if (o == q || o == k || o == v) return ATTN_ERR_INVALID_ARG;
    const int64_t *const in[4] = {q_strides, k_strides, v_strides, o_strides};
    TensorStrides st[4];
    attn_status_t status = parse_strides(in, B, Hq, Hkv, N, N, D, dtype, st);
    if (status != ATTN_OK) return status;
    Ctx c;
    status = get_ctx(stream, &c);
    if (status != ATTN_OK) return status;
    const float sc = resolve_scale(scale, D);
    if (half_dtype(dtype) && tc_full_supported(B, Hq, N, N, D)) {
        status = tc_causal_gqa(c, dtype, q, k, v, o, B, Hq, Hkv, N, D, sc, st);
        if (status != ATTN_ERR_UNSUPPORTED) return status;
    }
    return simt_causal_gqa(c, dtype, q, k, v, o, B, Hq, Hkv, N, D, sc, st);
}

attn_status_t attn_causal_gqa_fwd(const void *q, const void *k, const void *v, void *o, int B,
                                  int Hq, int Hkv, int N, int D, attn_dtype_t dtype, float scale,
                                  void *stream) {
    if (!q || !k || !v || !o) return ATTN_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o))
        return ATTN_ERR_INVALID_ARG;
    if (B < 1 || Hq < 1 || Hkv < 1 || N < 1 || Hq % Hkv != 0 || !valid_d(D) || !valid_dtype(dtype))
        return ATTN_ERR_INVALID_ARG;
    if (!small_enough(N, D) || (long long)B * Hq > 65535) return ATTN_ERR_UNSUPPORTED;
    if (o == q || o == k || o == v) return ATTN_ERR_INVALID_ARG;
    Ctx c;
    attn_status_t st = get_ctx(stream, &c);
    if (st != ATTN_OK) return st;
    const float sc = resolve_scale(scale, D);
    if (half_dtype(dtype) && tc_full_supported(B, Hq, N, N, D)) {
        st = tc_causal_gqa(c, dtype, q, k, v, o, B, Hq, Hkv, N, D, sc);
        if (st != ATTN_ERR_UNSUPPORTED) return st;
    }
    return simt_causal_gqa(c, dtype, q, k, v, o, B, Hq, Hkv, N, D, sc);
}

size_t attn_rope_joint_workspace_bytes(int B, int H, int N, int D, attn_dtype_t dtype) {
    if (B < 1 || H < 1 || N < 1 || !valid_d(D) || !valid_dtype(dtype)) return 0;
    const size_t one = ((size_t(B) * H * N * D * elem_size(dtype)) + 255) & ~size_t(255);
    return 2 * one;
}

attn_status_t attn_rope_joint_fwd(const void *q, const void *k, const void *v, void *o, int B,
                                  int H, int N, int D, const int32_t *pos,
                                  const int axes_dim[4], float theta, attn_dtype_t dtype,
                                  float scale, void *workspace, size_t workspace_bytes,
                                  void *stream) {
    if (!q || !k || !v || !o || !pos || !axes_dim || !workspace) return ATTN_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) ||
        (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
        return ATTN_ERR_INVALID_ARG;
    if (B < 1 || H < 1 || N < 1 || !valid_d(D) || !valid_dtype(dtype)) return ATTN_ERR_INVALID_ARG;
    if (!(theta > 0.f) || !isfinite(theta)) return ATTN_ERR_INVALID_ARG;
    int sum = 0;
    for (int a = 0; a < 4; ++a) {
        if (axes_dim[a] < 0 || (axes_dim[a] & 1)) return ATTN_ERR_INVALID_ARG;
        sum += axes_dim[a];
    }
    if (sum != D) return ATTN_ERR_INVALID_ARG;
    if (o == q || o == k || o == v) return ATTN_ERR_INVALID_ARG;
    if (!small_enough(N, D) || (long long)B * H > 65535) return ATTN_ERR_UNSUPPORTED;
    const size_t need = attn_rope_joint_workspace_bytes(B, H, N, D, dtype);
    if (workspace_bytes < need) return ATTN_ERR_RESOURCE;
    Ctx c;
    attn_status_t st = get_ctx(stream, &c);
    if (st != ATTN_OK) return st;
    uint8_t *qr = static_cast<uint8_t *>(workspace);
    uint8_t *kr = qr + need / 2;
    st = rope_rotate_qk(c, dtype, q, k, qr, kr, B * H, N, D, pos, axes_dim, theta);
    if (st != ATTN_OK) return st;
    const float sc = resolve_scale(scale, D);
    if (half_dtype(dtype) && tc_full_supported(B, H, N, N, D)) {
        st = tc_full(c, dtype, qr, kr, v, o, B, H, N, N, D, sc);
        if (st != ATTN_ERR_UNSUPPORTED) return st;
    }
    return simt_full(c, dtype, qr, kr, v, o, B, H, N, N, D, sc);
}

size_t attn_decode_gqa_workspace_bytes(int B, int Hq, int Hkv, int Lmax, int D) {
    if (B < 1 || Hq < 1 || Hkv < 1 || Hq % Hkv != 0 || Hq / Hkv > 8 || Lmax < 1) return 0;
    return decode_workspace_bytes(B, Hq, Hkv, Lmax, D);
}

static attn_status_t decode_entry(const void *q, const void *k_cache, const void *v_cache,
                                  const int32_t *seq_len, void *o, int B, int Hq, int Hkv,
                                  int Lmax, int D, attn_dtype_t dtype, float scale,
                                  void *workspace, size_t workspace_bytes, void *stream,
                                  bool ring) {
    if (!q || !k_cache || !v_cache || !seq_len || !o || !workspace) return ATTN_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(o) ||
        (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
        return ATTN_ERR_INVALID_ARG;
    if (B < 1 || Hq < 1 || Hkv < 1 || Lmax < 1 || !valid_dtype(dtype) || !valid_d(D))
        return ATTN_ERR_INVALID_ARG;
    if (Hq % Hkv != 0) return ATTN_ERR_INVALID_ARG;
    if (!half_dtype(dtype) || D == 32 || Hq / Hkv > 8) return ATTN_ERR_UNSUPPORTED;
    if ((long long)Lmax * D >= (1ll << 31) || B > 65535 || Hkv > 65535)
        return ATTN_ERR_UNSUPPORTED;
    if (o == q || o == k_cache || o == v_cache) return ATTN_ERR_INVALID_ARG;
    if (workspace_bytes < attn_decode_gqa_workspace_bytes(B, Hq, Hkv, Lmax, D))
        return ATTN_ERR_RESOURCE;
    Ctx c;
    attn_status_t st = get_ctx(stream, &c);
    if (st != ATTN_OK) return st;
    return decode_gqa(c, dtype, q, k_cache, v_cache, seq_len, o, B, Hq, Hkv, Lmax, D,
                      resolve_scale(scale, D), workspace, workspace_bytes, ring);
}

attn_status_t attn_decode_gqa(const void *q, const void *k_cache, const void *v_cache,
                              const int32_t *seq_len, void *o, int B, int Hq, int Hkv, int Lmax,
                              int D, attn_dtype_t dtype, float scale, void *workspace,
                              size_t workspace_bytes, void *stream) {
    return decode_entry(q, k_cache, v_cache, seq_len, o, B, Hq, Hkv, Lmax, D, dtype, scale,
                        workspace, workspace_bytes, stream, false);
}

attn_status_t attn_decode_gqa_ring(const void *q, const void *k_cache, const void *v_cache,
                                   const int32_t *seq_len, void *o, int B, int Hq, int Hkv,
                                   int Lmax, int D, attn_dtype_t dtype, float scale,
                                   void *workspace, size_t workspace_bytes, void *stream) {
    return decode_entry(q, k_cache, v_cache, seq_len, o, B, Hq, Hkv, Lmax, D, dtype, scale,
                        workspace, workspace_bytes, stream, true);
}

static attn_status_t append_entry(void *k_cache, void *v_cache, const void *k_new,
                                  const void *v_new, int32_t *seq_len, int B, int Hkv, int Lmax,
                                  int D, attn_dtype_t dtype, int advance, void *stream, bool ring) {
    if (!k_cache || !v_cache || !k_new || !v_new || !seq_len) return ATTN_ERR_INVALID_ARG;
    if (!aligned16(k_cache) || !aligned16(v_cache) || !aligned16(k_new) || !aligned16(v_new))
        return ATTN_ERR_INVALID_ARG;
    if (B < 1 || Hkv < 1 || Lmax < 1 || !valid_d(D) || !valid_dtype(dtype)) return ATTN_ERR_INVALID_ARG;
    if (k_cache == v_cache || k_new == k_cache || v_new == v_cache) return ATTN_ERR_INVALID_ARG;
    if ((long long)Lmax * D >= (1ll << 31)) return ATTN_ERR_UNSUPPORTED;
    Ctx c;
    attn_status_t st = get_ctx(stream, &c);
    if (st != ATTN_OK) return st;
    return kv_append(c, dtype, k_cache, v_cache, k_new, v_new, seq_len, B, Hkv, Lmax, D, advance,
                     ring);
}

attn_status_t attn_kv_append(void *k_cache, void *v_cache, const void *k_new, const void *v_new,
                             int32_t *seq_len, int B, int Hkv, int Lmax, int D, attn_dtype_t dtype,
                             int advance, void *stream) {
    return append_entry(k_cache, v_cache, k_new, v_new, seq_len, B, Hkv, Lmax, D, dtype, advance,
                        stream, false);
}

attn_status_t attn_kv_append_ring(void *k_cache, void *v_cache, const void *k_new,
                                  const void *v_new, int32_t *seq_len, int B, int Hkv, int Lmax,
                                  int D, attn_dtype_t dtype, int advance, void *stream) {
    return append_entry(k_cache, v_cache, k_new, v_new, seq_len, B, Hkv, Lmax, D, dtype, advance,
                        stream, true);
}

static attn_status_t check_na(int T, int Hg, int W, const int kernel[3]) {
    if (!kernel || T < 1 || Hg < 1 || W < 1) return ATTN_ERR_INVALID_ARG;
    for (int a = 0; a < 3; ++a)
        if (kernel[a] < 1 || (kernel[a] & 1) == 0) return ATTN_ERR_INVALID_ARG;
    if ((long long)T * Hg * W * 128 >= (1ll << 31)) return ATTN_ERR_UNSUPPORTED;
    return ATTN_OK;
}

attn_status_t attn_na3d_fwd(const void *q, const void *k, const void *v, void *o, int B,
                            int heads, int T, int Hg, int W, int D, const int kernel[3],
                            attn_dtype_t dtype, float scale, void *stream) {
    if (!q || !k || !v || !o) return ATTN_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o))
        return ATTN_ERR_INVALID_ARG;
    attn_status_t st = check_na(T, Hg, W, kernel);
    if (st != ATTN_OK) return st;
    if (B < 1 || heads < 1 || !valid_d(D) || !valid_dtype(dtype)) return ATTN_ERR_INVALID_ARG;
    if ((long long)B * heads > 65535) return ATTN_ERR_UNSUPPORTED;
    if (o == q || o == k || o == v) return ATTN_ERR_INVALID_ARG;
    Ctx c;
    st = get_ctx(stream, &c);
    if (st != ATTN_OK) return st;
    const float sc = resolve_scale(scale, D);
    if (half_dtype(dtype) && tc_na3d_supported(B, heads, T, Hg, W, D, kernel)) {
        st = tc_na3d(c, dtype, q, k, v, o, B, heads, T, Hg, W, D, kernel, sc);
        if (st != ATTN_ERR_UNSUPPORTED) return st;
    }
    return simt_na3d(c, dtype, q, k, v, o, B, heads, T, Hg, W, D, kernel, sc);
}

attn_status_t attn_na3d_fwd_strided(const void *q, const void *k, const void *v, void *o, int B,
                                    int heads, int T, int Hg, int W, int D, const int kernel[3],
                                    const int64_t q_strides[3], const int64_t k_strides[3],
                                    const int64_t v_strides[3], const int64_t o_strides[3],
                                    attn_dtype_t dtype, float scale, void *stream) {
    if (!q || !k || !v || !o) return ATTN_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o))
        return ATTN_ERR_INVALID_ARG;
    attn_status_t st = check_na(T, Hg, W, kernel);
    if (st != ATTN_OK) return st;
    if (B < 1 || heads < 1 || !valid_d(D) || !valid_dtype(dtype)) return ATTN_ERR_INVALID_ARG;
    if ((long long)B * heads > 65535) return ATTN_ERR_UNSUPPORTED;
    if (o == q || o == k || o == v) return ATTN_ERR_INVALID_ARG;
    const int N = T * Hg * W;
    const int64_t *const in[4] = {q_strides, k_strides, v_strides, o_strides};
    TensorStrides sts[4];
    st = parse_strides(in, B, heads, heads, N, N, D, dtype, sts);
    if (st != ATTN_OK) return st;
    Ctx c;
    st = get_ctx(stream, &c);
    if (st != ATTN_OK) return st;
    const float sc = resolve_scale(scale, D);
    // The tensor-core kernel addresses the contiguous layout only (its output
    // stores stay contiguous so that the dense path pays nothing for views);
    // any other layout runs on the exact SIMT kernel, which takes the strides.
    const long long n = N;
    bool dense = true;
    for (int i = 0; i < 4; ++i) {
        const TensorStrides d{(B == 1 ? D : heads * n * D), (heads == 1 ? D : n * D), D};
        dense = dense && sts[i].b == d.b && sts[i].h == d.h && sts[i].n == d.n;
    }
    if (dense && half_dtype(dtype) && tc_na3d_supported(B, heads, T, Hg, W, D, kernel)) {
        st = tc_na3d(c, dtype, q, k, v, o, B, heads, T, Hg, W, D, kernel, sc);
        if (st != ATTN_ERR_UNSUPPORTED) return st;
    }
    return simt_na3d(c, dtype, q, k, v, o, B, heads, T, Hg, W, D, kernel, sc, sts);
}

attn_status_t attn_na3d_window_starts(int T, int Hg, int W, const int kernel[3], int32_t *starts,
                                      void *stream) {
    if (!starts) return ATTN_ERR_INVALID_ARG;
    attn_status_t st = check_na(T, Hg, W, kernel);
    if (st != ATTN_OK) return st;
    Ctx c;
    st = get_ctx(stream, &c);
    if (st != ATTN_OK) return st;
    return na_starts(c, T, Hg, W, kernel, starts);
}

attn_status_t attn_debug_wait_test(uint64_t limit_ns, void *stream) {
    if (limit_ns < 1000 || limit_ns > kWaitLimitNs) return ATTN_ERR_INVALID_ARG;
    Ctx c;
    attn_status_t st = get_ctx(stream, &c);
    if (st != ATTN_OK) return st;
    wait_test_kernel<<<1, 1, 0, c.stream>>>(limit_ns, c.err);
    return launch_status(kFamDebug);
}

attn_status_t attn_debug_tc_tile(const void *q, const void *k, const void *v, const void *P,
                                 float *S, float *O, int D, void *stream) {
    if (!q || !k || !v || !P || !S || !O) return ATTN_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(P)) return ATTN_ERR_INVALID_ARG;
    if (D != 64 && D != 128) return ATTN_ERR_INVALID_ARG;
    Ctx c;
    attn_status_t st = get_ctx(stream, &c);
    if (st != ATTN_OK) return st;
    return tc_selftest(c, q, k, v, P, S, O, D);
}

}  // extern "C"
