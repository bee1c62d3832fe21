// The extern "C" boundary of libtrit: argument validation on the host, then
// dispatch to the launchers.  Nothing is enqueued when validation fails.
#include <math.h>
#include <stdio.h>
#include <string.h>

#include <mutex>

#include "trit_internal.cuh"

namespace trit {

namespace {

thread_local char g_last_cuda_error[256] = "";

constexpr int kMaxDevices = 64;
int g_sm_count[kMaxDevices] = {0};
int g_dev_ok[kMaxDevices] = {0};   // 0 unknown, 1 sm_103, -1 other
std::mutex g_dev_mutex;

trit_status cuda_fail(cudaError_t e) {
    snprintf(g_last_cuda_error, sizeof g_last_cuda_error, "%s: %s", cudaGetErrorName(e),
             cudaGetErrorString(e));
    return TRIT_E_CUDA;
}

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

bool rows_ok(int64_t n) { return n >= 1 && n <= kMaxRows; }
bool cols_ok(int64_t k) { return k >= 1 && k <= kMaxK; }

// The library carries sm_103a code only.
trit_status check_device() {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e);
    if (dev < 0 || dev >= kMaxDevices) return TRIT_E_DEVICE;
    std::lock_guard<std::mutex> lock(g_dev_mutex);
    if (g_dev_ok[dev] == 0) {
        int major = 0, minor = 0, sms = 0;
        cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        g_sm_count[dev] = sms;
        g_dev_ok[dev] = (major == 10 && minor == 3) ? 1 : -1;
    }
    return g_dev_ok[dev] == 1 ? TRIT_OK : TRIT_E_DEVICE;
}

trit_status check_proj(const trit_proj &p) {
    if (!p.planes || !p.x_i8 || !p.x_scale || (!p.y_i32 && !p.y_f32) ||
        (p.flags & ~TRIT_PROJ_PLANES_READY) != 0)
        return TRIT_E_ARG;
    if (!aligned(p.planes, 16) || !aligned(p.x_i8, 16) || !aligned(p.x_scale, 4) ||
        !aligned(p.y_i32, 4) || !aligned(p.y_f32, 4))
        return TRIT_E_ARG;
    if (!rows_ok(p.M) || !rows_ok(p.N) || !cols_ok(p.K)) return TRIT_E_SHAPE;
    if (!isfinite(p.w_scale) || !(p.w_scale > 0.0f)) return TRIT_E_SCALE;
    return TRIT_OK;
}

ProjDev to_dev(const trit_proj &p) {
    ProjDev d;
    d.planes = reinterpret_cast<const uint4 *>(p.planes);
    d.x = p.x_i8;
    d.xf = nullptr;
    d.x_i8_out = nullptr;
    d.x_scale = p.x_scale;
    d.y_i32 = p.y_i32;
    d.y_f32 = p.y_f32;
    d.M = p.M;
    d.N = p.N;
    d.K = int32_t(p.K);
    d.B = int32_t(beats_per_row(p.K));
    d.w_scale = p.w_scale;
    d.x_scale_val = 0.0f;
    d.planes_ready = (p.flags & TRIT_PROJ_PLANES_READY) != 0;
    return d;
}

trit_status run_many(const trit_proj *list, int32_t count, uint32_t *err_flag, cudaStream_t s) {
    if (!list || count <= 0 || !err_flag || !aligned(err_flag, 4)) return TRIT_E_ARG;
    for (int32_t i = 0; i < count; ++i) {
        trit_status st = check_proj(list[i]);
        if (st != TRIT_OK) return st;
    }
    trit_status st = check_device();
    if (st != TRIT_OK) return st;
    static thread_local ProjDev one[TRIT_MAX_LIST_PER_LAUNCH];
    static thread_local ProjDev many[TRIT_MAX_LIST_PER_LAUNCH];
    static thread_local ProjDev skinny[TRIT_MAX_LIST_PER_LAUNCH];
    static thread_local ProjDev dense[TRIT_MAX_LIST_PER_LAUNCH];
    int n1 = 0, nm = 0, ns = 0, nd = 0;
    auto flush1 = [&]() -> cudaError_t {
        cudaError_t e = n1 ? launch_gemv_many(one, n1, err_flag, s) : cudaSuccess;
        n1 = 0;
        return e;
    };
    auto flushm = [&]() -> cudaError_t {
        cudaError_t e = nm ? launch_gemm_dp4a_many(many, nm, err_flag, s) : cudaSuccess;
        nm = 0;
        return e;
    };
    auto flushs = [&]() -> cudaError_t {
        cudaError_t e = ns ? launch_skinny_many(skinny, ns, err_flag, s) : cudaSuccess;
        ns = 0;
        return e;
    };
    auto flushd = [&]() -> cudaError_t {
        cudaError_t e = nd ? launch_prefill_many(dense, nd, err_flag, s) : cudaSuccess;
        nd = 0;
        return e;
    };
    for (int32_t i = 0; i < count; ++i) {
        cudaError_t e = cudaSuccess;
        const ProjDev d = to_dev(list[i]);
        if (d.M == 1) {
            one[n1++] = d;
            if (n1 == TRIT_MAX_LIST_PER_LAUNCH) e = flush1();
        } else if (skinny_supported(d)) {
            skinny[ns++] = d;
            if (ns == TRIT_MAX_LIST_PER_LAUNCH) e = flushs();
        } else if (prefill_supported(d)) {
            dense[nd++] = d;
            if (nd == TRIT_MAX_LIST_PER_LAUNCH) e = flushd();
        } else {
            many[nm++] = d;
            if (nm == TRIT_MAX_LIST_PER_LAUNCH) e = flushm();
        }
        if (e != cudaSuccess) return cuda_fail(e);
    }
    cudaError_t e = flush1();
    if (e == cudaSuccess) e = flushm();
    if (e == cudaSuccess) e = flushs();
    if (e == cudaSuccess) e = flushd();
    return e == cudaSuccess ? TRIT_OK : cuda_fail(e);
}

trit_status check_qproj(const trit_qproj &p) {
    if (!p.planes || !p.x || (!p.y_i32 && !p.y_f32) || (p.flags & ~TRIT_PROJ_PLANES_READY) != 0)
        return TRIT_E_ARG;
    if (!aligned(p.planes, 16) || !aligned(p.x, 4) || !aligned(p.x_i8, 16) ||
        !aligned(p.x_scale, 4) || !aligned(p.y_i32, 4) || !aligned(p.y_f32, 4))
        return TRIT_E_ARG;
    if (!rows_ok(p.N) || !cols_ok(p.K) || p.K > TRIT_MAX_FUSED_K) return TRIT_E_SHAPE;
    if (!isfinite(p.w_scale) || !(p.w_scale > 0.0f)) return TRIT_E_SCALE;
    return TRIT_OK;
}

ProjDev to_dev(const trit_qproj &p) {
    ProjDev d;
    d.planes = reinterpret_cast<const uint4 *>(p.planes);
    d.x = nullptr;
    d.xf = p.x;
    d.x_i8_out = p.x_i8;
    d.x_scale = p.x_scale;
    d.y_i32 = p.y_i32;
    d.y_f32 = p.y_f32;
    d.M = 1;
    d.N = p.N;
    d.K = int32_t(p.K);
    d.B = int32_t(beats_per_row(p.K));
    d.w_scale = p.w_scale;
    d.x_scale_val = 0.0f;
    d.planes_ready = (p.flags & TRIT_PROJ_PLANES_READY) != 0;
    return d;
}

}  // namespace

int device_sm_count() {
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 0 && dev < kMaxDevices && g_sm_count[dev] > 0) return g_sm_count[dev];
    int sms = 0;
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    return sms > 0 ? sms : 1;
}

// ---- MLP blocks in two launches ----------------------------------------------------

namespace {
trit_status check_mlp_block(const trit_mlp_block &b) {
    if (!b.gate_planes || !b.up_planes || !b.down_planes || !b.x || !b.x_scale || !b.a_gate ||
        !b.a_up || !b.tmax || (!b.y_i32 && !b.y_f32) || (b.flags & ~TRIT_PROJ_PLANES_READY) != 0)
        return TRIT_E_ARG;
    if (!aligned(b.gate_planes, 16) || !aligned(b.up_planes, 16) || !aligned(b.down_planes, 16) ||
        !aligned(b.x, 4) || !aligned(b.x_scale, 4) || !aligned(b.a_gate, 16) ||
        !aligned(b.a_up, 16) || !aligned(b.tmax, 16) || !aligned(b.h_i8, 16) ||
        !aligned(b.h_scale, 4) || !aligned(b.y_i32, 4) || !aligned(b.y_f32, 4))
        return TRIT_E_ARG;
    if (!cols_ok(b.K) || !rows_ok(b.F) || !cols_ok(b.F) || !rows_ok(b.N) ||
        b.K > TRIT_MAX_FUSED_K || b.F > TRIT_MAX_FUSED_K)
        return TRIT_E_SHAPE;
    for (float w : {b.w_gate, b.w_up, b.w_down})
        if (!isfinite(w) || !(w > 0.0f)) return TRIT_E_SCALE;
    return TRIT_OK;
}

MlpBlockDev mlp_to_dev(const trit_mlp_block &b) {
    const bool ready = (b.flags & TRIT_PROJ_PLANES_READY) != 0;
    auto proj = [&](const uint8_t *planes, int64_t N, int64_t K, float w) {
        ProjDev d;
        d.planes = reinterpret_cast<const uint4 *>(planes);
        d.x = nullptr;
        d.xf = nullptr;
        d.x_i8_out = nullptr;
        d.x_scale = nullptr;
        d.y_i32 = nullptr;
        d.y_f32 = nullptr;
        d.M = 1;
        d.N = N;
        d.K = int32_t(K);
        d.B = int32_t(beats_per_row(K));
        d.w_scale = w;
        d.x_scale_val = 0.0f;
        d.planes_ready = ready;
        return d;
    };
    MlpBlockDev m;
    m.gate = proj(b.gate_planes, b.F, b.K, b.w_gate);
    m.gate.xf = b.x;
    m.gate.x_scale = b.x_scale;
    m.gate.y_i32 = b.a_gate;
    m.up = proj(b.up_planes, b.F, b.K, b.w_up);
    m.up.xf = b.x;
    m.up.y_i32 = b.a_up;
    m.down = proj(b.down_planes, b.N, b.F, b.w_down);
    m.down.x_i8_out = b.h_i8;
    m.down.x_scale = b.h_scale;
    m.down.y_i32 = b.y_i32;
    m.down.y_f32 = b.y_f32;
    m.w_gate = b.w_gate;
    m.w_up = b.w_up;
    m.tmax = static_cast<uint64_t *>(b.tmax);
    return m;
}

template <typename Launch>
trit_status run_mlp_blocks(const trit_mlp_block *list, int32_t count, uint32_t *err_flag,
                           trit_stream_t stream, Launch launch) {
    if (!list || count <= 0 || !err_flag || !aligned(err_flag, 4)) return TRIT_E_ARG;
    for (int32_t i = 0; i < count; ++i) {
        const trit_status st = check_mlp_block(list[i]);
        if (st != TRIT_OK) return st;
    }
    trit_status st = check_device();
    if (st != TRIT_OK) return st;
    static thread_local MlpBlockDev buf[TRIT_MAX_LIST_PER_LAUNCH];
    const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    for (int32_t base = 0; base < count; base += TRIT_MAX_LIST_PER_LAUNCH) {
        const int n = count - base < TRIT_MAX_LIST_PER_LAUNCH ? count - base : TRIT_MAX_LIST_PER_LAUNCH;
        for (int i = 0; i < n; ++i) buf[i] = mlp_to_dev(list[base + i]);
        const cudaError_t e = launch(buf, n, err_flag, s);
        if (e != cudaSuccess) return cuda_fail(e);
    }
    return TRIT_OK;
}
}  // namespace

}  // namespace trit

using namespace trit;

extern "C" {

TRIT_API const char *trit_status_string(trit_status s) {
    switch (s) {
        case TRIT_OK: return "TRIT_OK";
        case TRIT_E_ARG: return "TRIT_E_ARG: bad pointer, count or alignment";
        case TRIT_E_SHAPE: return "TRIT_E_SHAPE: size outside the supported range";
        case TRIT_E_SCALE: return "TRIT_E_SCALE: w_scale must be finite and > 0";
        case TRIT_E_CUDA: return "TRIT_E_CUDA: a CUDA call failed";
        case TRIT_E_DEVICE: return "TRIT_E_DEVICE: the current device is not sm_103";
        case TRIT_E_SCRATCH:
            return "TRIT_E_SCRATCH: the product needs more than TRIT_NOALLOC_SCRATCH_BYTES of scratch";
        case TRIT_E_VALUE: return "TRIT_E_VALUE: a weight outside {-1, 0, +1}";
    }
    return "unknown trit_status";
}

TRIT_API const char *trit_last_cuda_error(void) { return g_last_cuda_error; }

TRIT_API int32_t trit_abi_version(void) { return 4; }

TRIT_API int64_t trit_payload_bytes(int64_t N, int64_t K) {
    if (!rows_ok(N) || !cols_ok(K)) return -1;
    return N * beats_per_row(K) * 16;
}

TRIT_API trit_status trit_pack(const int8_t *w, int64_t N, int64_t K, float w_scale,
                               uint8_t *planes, float *scale_out, uint32_t *err_flag,
                               trit_stream_t stream) {
    if (!w || !planes || !err_flag || !aligned(planes, 16) || !aligned(scale_out, 4) ||
        !aligned(err_flag, 4))
        return TRIT_E_ARG;
    if (!rows_ok(N) || !cols_ok(K)) return TRIT_E_SHAPE;
    if (!isfinite(w_scale) || !(w_scale > 0.0f)) return TRIT_E_SCALE;
    trit_status st = check_device();
    if (st != TRIT_OK) return st;
    cudaError_t e = launch_pack(w, N, K, w_scale, planes, scale_out, err_flag,
                                reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? TRIT_OK : cuda_fail(e);
}

TRIT_API trit_status trit_unpack(const uint8_t *planes, int64_t N, int64_t K, int8_t *w,
                                 uint32_t *err_flag, trit_stream_t stream) {
    if (!w || !planes || !err_flag || !aligned(planes, 16) || !aligned(err_flag, 4))
        return TRIT_E_ARG;
    if (!rows_ok(N) || !cols_ok(K)) return TRIT_E_SHAPE;
    trit_status st = check_device();
    if (st != TRIT_OK) return st;
    cudaError_t e = launch_unpack(planes, N, K, w, err_flag, reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? TRIT_OK : cuda_fail(e);
}

TRIT_API trit_status trit_verify(const uint8_t *planes, int64_t N, int64_t K, uint32_t *err_flag,
                                 uint64_t *first_bad, trit_stream_t stream) {
    if (!planes || !err_flag || !aligned(planes, 16) || !aligned(err_flag, 4) ||
        !aligned(first_bad, 8))
        return TRIT_E_ARG;
    if (!rows_ok(N) || !cols_ok(K)) return TRIT_E_SHAPE;
    trit_status st = check_device();
    if (st != TRIT_OK) return st;
    cudaError_t e = launch_verify(planes, N, K, err_flag,
                                  reinterpret_cast<unsigned long long *>(first_bad),
                                  reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? TRIT_OK : cuda_fail(e);
}

TRIT_API trit_status trit_quant_act_many(const trit_act *list, int32_t count, uint32_t *err_flag,
                                         trit_stream_t stream) {
    if (!list || count <= 0 || !err_flag || !aligned(err_flag, 4)) return TRIT_E_ARG;
    int64_t rows = 0;
    for (int32_t i = 0; i < count; ++i) {
        const trit_act &a = list[i];
        if (!a.x || !a.x_i8 || !a.x_scale || !aligned(a.x, 4) || !aligned(a.x_i8, 16) ||
            !aligned(a.x_scale, 4))
            return TRIT_E_ARG;
        if (!rows_ok(a.M) || !cols_ok(a.K)) return TRIT_E_SHAPE;
        rows += a.M;
        if (rows > kMaxRows) return TRIT_E_SHAPE;
    }
    trit_status st = check_device();
    if (st != TRIT_OK) return st;
    cudaError_t e = launch_quant_many(list, count, err_flag, reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? TRIT_OK : cuda_fail(e);
}

TRIT_API trit_status trit_quant_act(const float *x, int64_t M, int64_t K, int8_t *x_i8,
                                    float *x_scale, uint32_t *err_flag, trit_stream_t stream) {
    trit_act a;
    a.x = x;
    a.x_i8 = x_i8;
    a.x_scale = x_scale;
    a.M = M;
    a.K = K;
    return trit_quant_act_many(&a, 1, err_flag, stream);
}

TRIT_API trit_status trit_gemm_many(const trit_proj *list, int32_t count, uint32_t *err_flag,
                                    trit_stream_t stream) {
    return run_many(list, count, err_flag, reinterpret_cast<cudaStream_t>(stream));
}

TRIT_API trit_status trit_quant_gemv_many(const trit_qproj *list, int32_t count, uint32_t *err_flag,
                                          trit_stream_t stream) {
    if (!list || count <= 0 || !err_flag || !aligned(err_flag, 4)) return TRIT_E_ARG;
    for (int32_t i = 0; i < count; ++i) {
        trit_status st = check_qproj(list[i]);
        if (st != TRIT_OK) return st;
    }
    trit_status st = check_device();
    if (st != TRIT_OK) return st;
    static thread_local ProjDev buf[TRIT_MAX_LIST_PER_LAUNCH];
    const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    for (int32_t base = 0; base < count; base += TRIT_MAX_LIST_PER_LAUNCH) {
        const int n = count - base < TRIT_MAX_LIST_PER_LAUNCH ? count - base : TRIT_MAX_LIST_PER_LAUNCH;
        for (int i = 0; i < n; ++i) buf[i] = to_dev(list[base + i]);
        cudaError_t e = launch_gemv_many(buf, n, err_flag, s);
        if (e != cudaSuccess) return cuda_fail(e);
    }
    return TRIT_OK;
}


TRIT_API int64_t trit_mlp_tmax_bytes(int64_t F) { return F < 1 ? 0 : mlp_tmax_bytes(F); }

TRIT_API trit_status trit_mlp_gate_up(const trit_mlp_block *list, int32_t count,
                                      uint32_t *err_flag, trit_stream_t stream) {
    return run_mlp_blocks(list, count, err_flag, stream, launch_mlp_gate_up);
}

TRIT_API trit_status trit_mlp_down(const trit_mlp_block *list, int32_t count,
                                   uint32_t *err_flag, trit_stream_t stream) {
    return run_mlp_blocks(list, count, err_flag, stream, launch_mlp_down);
}

TRIT_API trit_status trit_intmlp_gemv_many(const trit_mlpproj *list, int32_t count,
                                           uint32_t *err_flag, trit_stream_t stream) {
    if (!list || count <= 0 || !err_flag || !aligned(err_flag, 4)) return TRIT_E_ARG;
    for (int32_t i = 0; i < count; ++i) {
        const trit_mlpproj &p = list[i];
        if (!p.planes || !p.a_gate || !p.a_up || !p.x_scale || (!p.y_i32 && !p.y_f32) ||
            p.reserved != 0)
            return TRIT_E_ARG;
        if (!aligned(p.planes, 16) || !aligned(p.a_gate, 4) || !aligned(p.a_up, 4) ||
            !aligned(p.x_scale, 4) || !aligned(p.h_i8, 16) || !aligned(p.h_scale, 4) ||
            !aligned(p.y_i32, 4) || !aligned(p.y_f32, 4))
            return TRIT_E_ARG;
        if (!rows_ok(p.N) || !cols_ok(p.K) || p.K > TRIT_MAX_FUSED_K) return TRIT_E_SHAPE;
        for (float w : {p.w_scale, p.w_gate, p.w_up})
            if (!isfinite(w) || !(w > 0.0f)) return TRIT_E_SCALE;
    }
    trit_status st = check_device();
    if (st != TRIT_OK) return st;
    static thread_local MlpProjDev buf[TRIT_MAX_LIST_PER_LAUNCH];
    const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    for (int32_t base = 0; base < count; base += TRIT_MAX_LIST_PER_LAUNCH) {
        const int n = count - base < TRIT_MAX_LIST_PER_LAUNCH ? count - base : TRIT_MAX_LIST_PER_LAUNCH;
        for (int i = 0; i < n; ++i) {
            const trit_mlpproj &p = list[base + i];
            MlpProjDev &m = buf[i];
            m.down.planes = reinterpret_cast<const uint4 *>(p.planes);
            m.down.x = nullptr;
            m.down.xf = nullptr;
            m.down.x_i8_out = p.h_i8;
            m.down.x_scale = p.h_scale;
            m.down.y_i32 = p.y_i32;
            m.down.y_f32 = p.y_f32;
            m.down.M = 1;
            m.down.N = p.N;
            m.down.K = int32_t(p.K);
            m.down.B = int32_t(beats_per_row(p.K));
            m.down.w_scale = p.w_scale;
            m.down.x_scale_val = 0.0f;
            m.down.planes_ready = false;
            m.a_gate = p.a_gate;
            m.a_up = p.a_up;
            m.x_scale_in = p.x_scale;
            m.w_gate = p.w_gate;
            m.w_up = p.w_up;
        }
        cudaError_t e = launch_intmlp_gemv_many(buf, n, err_flag, s);
        if (e != cudaSuccess) return cuda_fail(e);
    }
    return TRIT_OK;
}

TRIT_API trit_status trit_gemm(const uint8_t *planes, float w_scale, const int8_t *x_i8,
                               const float *x_scale, int64_t M, int64_t N, int64_t K,
                               int32_t *y_i32, float *y_f32, uint32_t *err_flag,
                               trit_stream_t stream) {
    trit_proj p;
    p.planes = planes;
    p.x_i8 = x_i8;
    p.x_scale = x_scale;
    p.y_i32 = y_i32;
    p.y_f32 = y_f32;
    p.M = M;
    p.N = N;
    p.K = K;
    p.w_scale = w_scale;
    p.flags = 0;
    return run_many(&p, 1, err_flag, reinterpret_cast<cudaStream_t>(stream));
}

TRIT_API trit_status trit_gemv(const uint8_t *planes, float w_scale, const int8_t *x_i8,
                               float x_scale, int64_t N, int64_t K, int32_t *y_i32, float *y_f32,
                               uint32_t *err_flag, trit_stream_t stream) {
    // validated as trit_gemm validates M = 1, with the scale checked here: the
    // kernel takes it as a launch parameter instead of reading it from memory
    trit_proj p;
    p.planes = planes;
    p.x_i8 = x_i8;
    p.x_scale = reinterpret_cast<const float *>(planes);   // any non-NULL aligned stand-in
    p.y_i32 = y_i32;
    p.y_f32 = y_f32;
    p.M = 1;
    p.N = N;
    p.K = K;
    p.w_scale = w_scale;
    p.flags = 0;
    if (!err_flag || !aligned(err_flag, 4)) return TRIT_E_ARG;
    trit_status st = check_proj(p);
    if (st != TRIT_OK) return st;
    if (!isfinite(x_scale) || x_scale < 0.0f) return TRIT_E_SCALE;
    st = check_device();
    if (st != TRIT_OK) return st;
    ProjDev d = to_dev(p);
    d.x_scale = nullptr;
    d.x_scale_val = x_scale;
    cudaError_t e = launch_gemv_many(&d, 1, err_flag, reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? TRIT_OK : cuda_fail(e);
}

TRIT_API trit_status trit_quant_act_folded(const float *x, const float *gain, int64_t M, int64_t K,
                                           float eps, int8_t *x_i8, float *x_scale,
                                           uint32_t *err_flag, trit_stream_t stream) {
    if (!x || !gain || !x_i8 || !x_scale || !err_flag || !aligned(x, 4) || !aligned(gain, 4) ||
        !aligned(x_i8, 16) || !aligned(x_scale, 4) || !aligned(err_flag, 4))
        return TRIT_E_ARG;
    if (!rows_ok(M) || !cols_ok(K)) return TRIT_E_SHAPE;
    if (!isfinite(eps) || eps < 0.0f) return TRIT_E_SCALE;
    trit_status st = check_device();
    if (st != TRIT_OK) return st;
    cudaError_t e = launch_quant_folded(x, gain, M, K, eps, x_i8, x_scale, err_flag,
                                        reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? TRIT_OK : cuda_fail(e);
}

TRIT_API trit_status trit_read_probe(const void *buf, int64_t bytes, uint32_t *sink,
                                     trit_stream_t stream) {
    if (!buf || !sink || !aligned(buf, 16) || !aligned(sink, 4) || bytes < 16 || bytes % 16)
        return TRIT_E_ARG;
    trit_status st = check_device();
    if (st != TRIT_OK) return st;
    cudaError_t e = launch_read_probe(buf, bytes, sink, reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? TRIT_OK : cuda_fail(e);
}

TRIT_API trit_status trit_issue_probe(int32_t kind, int32_t blocks, int32_t threads, int64_t iters,
                                      uint32_t *sink, uint64_t *rec, trit_stream_t stream) {
    if (!sink || !rec || !aligned(sink, 4) || !aligned(rec, 8)) return TRIT_E_ARG;
    if (kind < TRIT_PROBE_DP4A || kind > TRIT_PROBE_DP4A_SU || blocks < 1 || threads < 32 ||
        threads > 512 || threads % 32 || iters < 1)
        return TRIT_E_ARG;
    trit_status st = check_device();
    if (st != TRIT_OK) return st;
    cudaError_t e = launch_issue_probe(kind, blocks, threads, iters, sink,
                                       reinterpret_cast<unsigned long long *>(rec),
                                       reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? TRIT_OK : cuda_fail(e);
}

TRIT_API trit_status trit_check_div127(uint64_t *mismatches) {
    if (!mismatches) return TRIT_E_ARG;
    *mismatches = ~uint64_t(0);
    trit_status st = check_device();
    if (st != TRIT_OK) return st;
    unsigned long long *d = nullptr;
    cudaError_t e = cudaMalloc(reinterpret_cast<void **>(&d), sizeof(unsigned long long));
    if (e != cudaSuccess) return cuda_fail(e);
    e = cudaMemset(d, 0, sizeof(unsigned long long));
    if (e == cudaSuccess) e = launch_check_div127(0, uint64_t(1) << 32, d, 0);
    unsigned long long h = 0;
    if (e == cudaSuccess) e = cudaMemcpy(&h, d, sizeof(h), cudaMemcpyDeviceToHost);
    cudaFree(d);
    if (e != cudaSuccess) return cuda_fail(e);
    *mismatches = h;
    return TRIT_OK;
}

TRIT_API trit_status trit_intmlp_quant(const int32_t *a_gate, const int32_t *a_up, int64_t M,
                                       int64_t N, float w_scale_gate, float w_scale_up,
                                       const float *x_scale, int8_t *h_i8, float *h_scale,
                                       trit_stream_t stream) {
    if (!a_gate || !a_up || !x_scale || !h_i8 || !h_scale || !aligned(a_gate, 4) ||
        !aligned(a_up, 4) || !aligned(x_scale, 4) || !aligned(h_i8, 16) || !aligned(h_scale, 4))
        return TRIT_E_ARG;
    if (!rows_ok(M) || !cols_ok(N)) return TRIT_E_SHAPE;
    if (!isfinite(w_scale_gate) || !(w_scale_gate > 0.0f) || !isfinite(w_scale_up) ||
        !(w_scale_up > 0.0f))
        return TRIT_E_SCALE;
    trit_status st = check_device();
    if (st != TRIT_OK) return st;
    cudaError_t e = launch_intmlp_quant(a_gate, a_up, M, N, w_scale_gate, w_scale_up, x_scale, h_i8,
                                        h_scale, reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? TRIT_OK : cuda_fail(e);
}

TRIT_API trit_status trit_gemm_noalloc(const uint8_t *planes, float w_scale, const int8_t *x_i8,
                                       const float *x_scale, int64_t M, int64_t N, int64_t K,
                                       int32_t *y_i32, float *y_f32, uint32_t *err_flag,
                                       trit_stream_t stream) {
    trit_proj p;
    p.planes = planes;
    p.x_i8 = x_i8;
    p.x_scale = x_scale;
    p.y_i32 = y_i32;
    p.y_f32 = y_f32;
    p.M = M;
    p.N = N;
    p.K = K;
    p.w_scale = w_scale;
    p.flags = 0;
    const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (!err_flag || !aligned(err_flag, 4)) return TRIT_E_ARG;
    trit_status st = check_proj(p);
    if (st != TRIT_OK) return st;
    const ProjDev d = to_dev(p);
    // Only the tensor-core paths use scratch; the others allocate nothing.
    const bool small = skinny_supported(d);
    if (!small && !prefill_supported(d)) return run_many(&p, 1, err_flag, s);
    const int64_t need = small ? skinny_scratch_bytes(d) : prefill_scratch_bytes(d);
    if (need > TRIT_NOALLOC_SCRATCH_BYTES) return TRIT_E_SCRATCH;
    st = check_device();
    if (st != TRIT_OK) return st;
    uint8_t *xh = nullptr;
    cudaError_t e = fixed_scratch(&xh);
    if (e == cudaSuccess)
        e = small ? launch_skinny_into(d, xh, err_flag, s) : launch_prefill_into(d, xh, err_flag, s);
    return e == cudaSuccess ? TRIT_OK : cuda_fail(e);
}

TRIT_API trit_status trit_bitcos_pack(const int8_t *w, int64_t N, int64_t K, uint64_t *bitmap,
                                      uint32_t *sign_off, uint32_t *signs, int64_t *sign_words) {
    if (!w || !sign_words) return TRIT_E_ARG;
    if (signs && (!bitmap || !sign_off)) return TRIT_E_ARG;
    if (!rows_ok(N) || K < 1 || K > kBitcosMaxK) return TRIT_E_SHAPE;
    return static_cast<trit_status>(bitcos_pack_host(w, N, K, bitmap, sign_off, signs, sign_words));
}

TRIT_API trit_status trit_bitcos_gemv_many(const trit_bitcos_proj *list, int32_t count,
                                           trit_stream_t stream) {
    if (!list || count <= 0) return TRIT_E_ARG;
    for (int32_t i = 0; i < count; ++i) {
        const trit_bitcos_proj &p = list[i];
        if (!p.bitmap || !p.sign_off || !p.signs || !p.x_i8 || !p.x_scale || (!p.y_i32 && !p.y_f32) ||
            p.reserved != 0)
            return TRIT_E_ARG;
        if (!aligned(p.bitmap, 16) || !aligned(p.sign_off, 4) || !aligned(p.signs, 4) ||
            !aligned(p.x_i8, 16) || !aligned(p.x_scale, 4) || !aligned(p.y_i32, 4) ||
            !aligned(p.y_f32, 4))
            return TRIT_E_ARG;
        if (!rows_ok(p.N) || p.K < 1 || p.K > kBitcosMaxK || p.sign_words < 2) return TRIT_E_SHAPE;
        if (!isfinite(p.w_scale) || !(p.w_scale > 0.0f)) return TRIT_E_SCALE;
    }
    trit_status st = check_device();
    if (st != TRIT_OK) return st;
    static thread_local BitcosDev devs[TRIT_MAX_LIST_PER_LAUNCH];
    const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    for (int32_t base = 0; base < count; base += TRIT_MAX_LIST_PER_LAUNCH) {
        const int n = count - base < TRIT_MAX_LIST_PER_LAUNCH ? count - base : TRIT_MAX_LIST_PER_LAUNCH;
        for (int i = 0; i < n; ++i) {
            const trit_bitcos_proj &p = list[base + i];
            BitcosDev &d = devs[i];
            d.bitmap = p.bitmap;
            d.sign_off = p.sign_off;
            d.signs = p.signs;
            d.x = p.x_i8;
            d.x_scale = p.x_scale;
            d.y_i32 = p.y_i32;
            d.y_f32 = p.y_f32;
            d.N = p.N;
            d.K = p.K;
            d.sign_words = p.sign_words;
            d.w_scale = p.w_scale;
        }
        const cudaError_t e = launch_bitcos_many(devs, n, s);
        if (e != cudaSuccess) return cuda_fail(e);
    }
    return TRIT_OK;
}

}  // extern "C"
