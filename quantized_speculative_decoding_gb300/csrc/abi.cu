// C ABI of libsd.so (declared in include/sd.h): argument checks, host-side
// fault injection, per-device / per-stream workspace, dispatch to kernels.
#include <cmath>
#include <cstdlib>
#include <cstring>
#include <map>
#include <mutex>
#include <tuple>
#include <utility>

#include "../../include/sd.h"
#include "sd_internal.h"

extern "C" sd_status sd_w4_pack_impl(const float* w, int N, int K, int group, uint32_t* qweight,
                                     uint16_t* scales, uint16_t* zeros);
extern "C" sd_status sd_w8_pack_impl(const float* w, int N, int K, int8_t* qweight,
                                     uint16_t* scales);
extern "C" sd_status sd_wb_pack_impl(const float* w, int N, int K, int group, int bits, uint32_t* packed,
                                     uint16_t* scales, uint16_t* zeros);

namespace sd {
namespace {

std::mutex g_mu;
std::map<int, int*> g_err_words;
std::map<int, int> g_sms;

struct Workspace {
    void* ptr = nullptr;
    size_t bytes = 0;
};
// workspaces keyed by (purpose, device, stream); purpose 0 = verify, 1 = W4A16 split-K, 2 = sample
std::map<std::tuple<int, int, cudaStream_t>, Workspace> g_ws;

// Returns a zero-initialised (on first allocation) workspace of at least
// `need` bytes for (purpose, device, stream), or nullptr on failure.  Growing
// synchronises the stream before the old buffer is freed.
void* workspace(int purpose, int dev, cudaStream_t s, size_t need) {
    std::lock_guard<std::mutex> lk(g_mu);
    Workspace& w = g_ws[std::make_tuple(purpose, dev, s)];
    if (w.bytes >= need) return w.ptr;
    if (w.ptr) {
        if (cudaStreamSynchronize(s) != cudaSuccess) return nullptr;
        cudaFree(w.ptr);
        w.ptr = nullptr;
        w.bytes = 0;
    }
    void* p = nullptr;
    if (cudaMalloc(&p, need) != cudaSuccess) return nullptr;
    if (cudaMemsetAsync(p, 0, need, s) != cudaSuccess) {
        cudaFree(p);
        return nullptr;
    }
    w.ptr = p;
    w.bytes = need;
    return p;
}

// Dedicated, zero-initialised uint32 counters for (purpose, device, stream).
// They are never used for anything else, and every kernel that uses them
// leaves them at zero when it completes (atomicInc wraps), so later calls
// with other sizes find them at zero.  Growing synchronises the stream first.
std::map<std::tuple<int, int, cudaStream_t>, Workspace> g_counters;

unsigned* counters(int purpose, int dev, cudaStream_t s, size_t n) {
    std::lock_guard<std::mutex> lk(g_mu);
    Workspace& w = g_counters[std::make_tuple(purpose, dev, s)];
    const size_t need = n * sizeof(unsigned);
    if (w.bytes >= need) return static_cast<unsigned*>(w.ptr);
    if (w.ptr) {
        if (cudaStreamSynchronize(s) != cudaSuccess) return nullptr;
        cudaFree(w.ptr);
        w.ptr = nullptr;
        w.bytes = 0;
    }
    size_t bytes = 4096;
    while (bytes < need) bytes *= 2;
    void* p = nullptr;
    if (cudaMalloc(&p, bytes) != cudaSuccess) return nullptr;
    if (cudaMemsetAsync(p, 0, bytes, s) != cudaSuccess) {
        cudaFree(p);
        return nullptr;
    }
    w.ptr = p;
    w.bytes = bytes;
    return static_cast<unsigned*>(p);
}

// Kernel family of the row-major W4A16 linear: automatic (the register-operand
// mma.sync kernel on the row-major layout for M <= 32 where its alignment and
// K rules hold, else the CUDA-core GEMV at M = 1 and the tcgen05 kernels from
// M = 2; the batched tcgen05 kernel above M = 32), or one family forced by the
// test hook sd_test_w4a16_linear_path.
enum LinearPath { kPathAuto = 0, kPathCudaCore = 1, kPathTensorCore = 2, kPathMma = 3 };

// SD_FAULT_INJECT="name:status[,name:status...]" -> the status for `name`, or 0.
int injected(const char* name) {
    const char* env = std::getenv("SD_FAULT_INJECT");
    if (!env || !*env) return 0;
    const size_t n = std::strlen(name);
    const char* p = env;
    while (*p) {
        const char* colon = std::strchr(p, ':');
        if (!colon) break;
        const char* end = std::strchr(colon, ',');
        if ((size_t)(colon - p) == n && std::strncmp(p, name, n) == 0) {
            const int code = std::atoi(colon + 1);
            return code;
        }
        if (!end) break;
        p = end + 1;
    }
    return 0;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

sd_status from_cuda(cudaError_t e) { return e == cudaSuccess ? SD_OK : SD_ERR_CUDA; }

}  // namespace

int* device_error_word(int device) {
    std::lock_guard<std::mutex> lk(g_mu);
    auto it = g_err_words.find(device);
    if (it != g_err_words.end()) return it->second;
    int* p = nullptr;
    if (cudaMalloc(&p, sizeof(int)) != cudaSuccess) return nullptr;
    if (cudaMemset(p, 0, sizeof(int)) != cudaSuccess) {
        cudaFree(p);
        return nullptr;
    }
    g_err_words[device] = p;
    return p;
}

int num_sms(int device) {
    {
        std::lock_guard<std::mutex> lk(g_mu);
        auto it = g_sms.find(device);
        if (it != g_sms.end()) return it->second;
    }
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, device) != cudaSuccess || n <= 0)
        n = 148;
    std::lock_guard<std::mutex> lk(g_mu);
    g_sms[device] = n;
    return n;
}

}  // namespace sd

using namespace sd;

#define SD_INJECT(name)                        \
    do {                                       \
        const int _c = injected(name);         \
        if (_c) return (sd_status)_c;          \
    } while (0)

#define SD_GUARD_BEGIN try {
#define SD_GUARD_END \
    }                \
    catch (...) {    \
        return SD_ERR_INTERNAL; \
    }

extern "C" {

const char* sd_status_string(int status) {
    switch (status) {
        case SD_OK: return "SD_OK";
        case SD_ERR_INVALID_ARG: return "SD_ERR_INVALID_ARG";
        case SD_ERR_UNSUPPORTED: return "SD_ERR_UNSUPPORTED";
        case SD_ERR_CUDA: return "SD_ERR_CUDA";
        case SD_ERR_TIMEOUT: return "SD_ERR_TIMEOUT";
        case SD_ERR_INTERNAL: return "SD_ERR_INTERNAL";
        default: return "SD_ERR_UNKNOWN";
    }
}

int sd_version(void) { return (1 << 16) | 0; }

sd_status sd_w4_pack(const float* w, int N, int K, int group, uint32_t* qweight,
                     uint16_t* scales, uint16_t* zeros) {
    SD_INJECT("sd_w4_pack");
    SD_GUARD_BEGIN
    return sd_w4_pack_impl(w, N, K, group, qweight, scales, zeros);
    SD_GUARD_END
}

sd_status sd_wb_pack(const float* w, int N, int K, int group, int bits, uint32_t* packed,
                     uint16_t* scales, uint16_t* zeros) {
    SD_INJECT("sd_wb_pack");
    SD_GUARD_BEGIN
    return sd_wb_pack_impl(w, N, K, group, bits, packed, scales, zeros);
    SD_GUARD_END
}

sd_status sd_w8_pack(const float* w, int N, int K, int8_t* qweight, uint16_t* scales) {
    SD_INJECT("sd_w8_pack");
    SD_GUARD_BEGIN
    return sd_w8_pack_impl(w, N, K, qweight, scales);
    SD_GUARD_END
}

}  // extern "C"

namespace {
sd_status w4a16_linear_impl(const void* x, const uint32_t* qweight, const void* scales, const void* zeros,
                            int group, int M, int N, int K, void* out, void* stream, int path) {
    if (!x || !qweight || !scales || !zeros || !out) return SD_ERR_INVALID_ARG;
    if (M <= 0 || N <= 0 || K <= 0 || group <= 0 || K % 8 != 0 || K % group != 0)
        return SD_ERR_INVALID_ARG;
    if (!aligned(x, 16) || !aligned(qweight, 16) || !aligned(scales, 2) || !aligned(zeros, 2) ||
        !aligned(out, 2))
        return SD_ERR_INVALID_ARG;
    if (group != 128) return SD_ERR_UNSUPPORTED;
    if (path == kPathCudaCore && M > 8) return SD_ERR_UNSUPPORTED;
    const bool mma_ok = w4a16_mma_rowmajor_ok(qweight, scales, zeros, M, K);
    if (path == kPathMma && !mma_ok) return SD_ERR_UNSUPPORTED;
    SD_GUARD_BEGIN
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return SD_ERR_CUDA;
    const int sms = num_sms(dev);
    if (path == kPathMma || (path == kPathAuto && mma_ok))
        return from_cuda(launch_w4a16_mma_rowmajor(x, qweight, scales, zeros, M, N, K, out, sms, s));
    if (path == kPathCudaCore || (path == kPathAuto && M < 2))
        return from_cuda(launch_gemv(0, x, qweight, scales, zeros, M, N, K, out, s));
    int* err = device_error_word(dev);
    if (!err) return SD_ERR_CUDA;
    if (M <= 32) {
        // small M: TMEM-dequant kernel
        const size_t need2 = w4a16_tc2_workspace_bytes(M, N, K, sms);
        void* ws2 = nullptr;
        unsigned* cnt2 = nullptr;
        if (need2) {
            ws2 = workspace(1, dev, s, need2);
            cnt2 = counters(1, dev, s, (size_t)(N + 127) / 128);
            if (!ws2 || !cnt2) return SD_ERR_CUDA;
        }
        return from_cuda(launch_w4a16_tc2(x, qweight, scales, zeros, M, N, K, out, ws2, need2,
                                          cnt2, sms, err, s));
    }
    // blocks of at most 160 rows of x (the MMA's N extent in the batched kernel)
    const int mb_max = M < 160 ? M : 160;
    const size_t need = w4a16_tc_workspace_bytes(mb_max, N, K, sms);
    void* ws = nullptr;
    unsigned* cnt = nullptr;
    if (need) {
        ws = workspace(1, dev, s, need);
        cnt = counters(1, dev, s, (size_t)(N + 127) / 128);
        if (!ws || !cnt) return SD_ERR_CUDA;
    }
    for (int m0 = 0; m0 < M; m0 += 160) {
        const int mb = M - m0 < 160 ? M - m0 : 160;
        const cudaError_t e = launch_w4a16_tc(
            static_cast<const char*>(x) + (size_t)m0 * K * 2, qweight, scales, zeros, mb, N, K,
            static_cast<char*>(out) + (size_t)m0 * N * 2, ws, need, cnt, sms, err, s);
        if (e != cudaSuccess) return SD_ERR_CUDA;
    }
    return SD_OK;
    SD_GUARD_END
}
}  // namespace

extern "C" {

sd_status sd_w4a16_linear(const void* x, const uint32_t* qweight, const void* scales,
                          const void* zeros, int group, int M, int N, int K, void* out,
                          void* stream) {
    SD_INJECT("sd_w4a16_linear");
    return w4a16_linear_impl(x, qweight, scales, zeros, group, M, N, K, out, stream, kPathAuto);
}

sd_status sd_test_w4a16_linear_path(const void* x, const uint32_t* qweight, const void* scales,
                                    const void* zeros, int group, int M, int N, int K, void* out, int path,
                                    void* stream) {
    SD_INJECT("sd_test_w4a16_linear_path");
    if (path != kPathCudaCore && path != kPathTensorCore && path != kPathMma) return SD_ERR_INVALID_ARG;
    return w4a16_linear_impl(x, qweight, scales, zeros, group, M, N, K, out, stream, path);
}

sd_status sd_w4_tiled_bytes(int N, int K, int group, size_t* qweight_bytes, size_t* sz_bytes) {
    SD_INJECT("sd_w4_tiled_bytes");
    if (!qweight_bytes || !sz_bytes || N <= 0 || K <= 0 || group <= 0 || K % group != 0)
        return SD_ERR_INVALID_ARG;
    if (group != 128) return SD_ERR_UNSUPPORTED;
    w4_tiled_sizes(N, K, qweight_bytes, sz_bytes);
    return SD_OK;
}

sd_status sd_w4_tile(const uint32_t* qweight, const void* scales, const void* zeros, int group,
                     int N, int K, void* tiled_qweight, void* tiled_sz, void* stream) {
    SD_INJECT("sd_w4_tile");
    if (!qweight || !scales || !zeros || !tiled_qweight || !tiled_sz) return SD_ERR_INVALID_ARG;
    if (N <= 0 || K <= 0 || group <= 0 || K % group != 0) return SD_ERR_INVALID_ARG;
    if (!aligned(qweight, 16) || !aligned(tiled_qweight, 16) || !aligned(scales, 2) ||
        !aligned(zeros, 2) || !aligned(tiled_sz, 16))
        return SD_ERR_INVALID_ARG;
    if (group != 128) return SD_ERR_UNSUPPORTED;
    SD_GUARD_BEGIN
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return SD_ERR_CUDA;
    int* err = device_error_word(dev);
    if (!err) return SD_ERR_CUDA;
    return from_cuda(launch_w4_tile(qweight, scales, zeros, N, K, tiled_qweight, tiled_sz, err,
                                    num_sms(dev), static_cast<cudaStream_t>(stream)));
    SD_GUARD_END
}

sd_status sd_w4a16_linear_tiled(const void* x, const void* tiled_qweight, const void* tiled_sz,
                                int group, int M, int N, int K, void* out, void* stream) {
    SD_INJECT("sd_w4a16_linear_tiled");
    if (!x || !tiled_qweight || !tiled_sz || !out) return SD_ERR_INVALID_ARG;
    if (M <= 0 || N <= 0 || K <= 0 || group <= 0 || K % 8 != 0 || K % group != 0)
        return SD_ERR_INVALID_ARG;
    if (!aligned(x, 16) || !aligned(tiled_qweight, 16) || !aligned(tiled_sz, 16) || !aligned(out, 2))
        return SD_ERR_INVALID_ARG;
    if (group != 128) return SD_ERR_UNSUPPORTED;
    SD_GUARD_BEGIN
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return SD_ERR_CUDA;
    const int sms = num_sms(dev);
    // blocks of at most 32 rows of x
    for (int m0 = 0; m0 < M; m0 += 32) {
        const int mb = M - m0 < 32 ? M - m0 : 32;
        const cudaError_t e = launch_w4a16_mma(static_cast<const char*>(x) + (size_t)m0 * K * 2,
                                               tiled_qweight, tiled_sz, mb, N, K,
                                               static_cast<char*>(out) + (size_t)m0 * N * 2, sms, s);
        if (e != cudaSuccess) return SD_ERR_CUDA;
    }
    return SD_OK;
    SD_GUARD_END
}

sd_status sd_wb_tiled_bytes(int N, int K, int group, int bits, size_t* qweight_bytes, size_t* sz_bytes) {
    SD_INJECT("sd_wb_tiled_bytes");
    if (!qweight_bytes || !sz_bytes || N <= 0 || K <= 0 || group <= 0 || K % group != 0) return SD_ERR_INVALID_ARG;
    if (bits < 2 || bits > 4) return SD_ERR_INVALID_ARG;
    if (group != 128) return SD_ERR_UNSUPPORTED;
    wb_tiled_sizes(N, K, bits, qweight_bytes, sz_bytes);
    return SD_OK;
}

sd_status sd_wb_tile(const uint32_t* packed, const void* scales, const void* zeros, int group, int bits, int N,
                     int K, void* tiled_qweight, void* tiled_sz, void* stream) {
    SD_INJECT("sd_wb_tile");
    if (!packed || !scales || !zeros || !tiled_qweight || !tiled_sz) return SD_ERR_INVALID_ARG;
    if (N <= 0 || K <= 0 || group <= 0 || K % group != 0 || bits < 2 || bits > 4) return SD_ERR_INVALID_ARG;
    if (!aligned(packed, 4) || !aligned(tiled_qweight, 16) || !aligned(scales, 2) || !aligned(zeros, 2) ||
        !aligned(tiled_sz, 16))
        return SD_ERR_INVALID_ARG;
    if (group != 128) return SD_ERR_UNSUPPORTED;
    if (bits == 4)  // the 4-bit stream is the sd_w4_pack layout
        return sd_w4_tile(packed, scales, zeros, group, N, K, tiled_qweight, tiled_sz, stream);
    SD_GUARD_BEGIN
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return SD_ERR_CUDA;
    int* err = device_error_word(dev);
    if (!err) return SD_ERR_CUDA;
    return from_cuda(launch_wb_tile(packed, scales, zeros, bits, N, K, tiled_qweight, tiled_sz, err, num_sms(dev),
                                    static_cast<cudaStream_t>(stream)));
    SD_GUARD_END
}

sd_status sd_wb_linear_tiled(const void* x, const void* tiled_qweight, const void* tiled_sz, int group, int bits,
                             int M, int N, int K, void* out, void* stream) {
    SD_INJECT("sd_wb_linear_tiled");
    if (!x || !tiled_qweight || !tiled_sz || !out) return SD_ERR_INVALID_ARG;
    if (M <= 0 || N <= 0 || K <= 0 || group <= 0 || K % group != 0 || bits < 2 || bits > 4)
        return SD_ERR_INVALID_ARG;
    if (!aligned(x, 16) || !aligned(tiled_qweight, 16) || !aligned(tiled_sz, 16) || !aligned(out, 2))
        return SD_ERR_INVALID_ARG;
    if (group != 128) return SD_ERR_UNSUPPORTED;
    if (bits == 4) return sd_w4a16_linear_tiled(x, tiled_qweight, tiled_sz, group, M, N, K, out, stream);
    SD_GUARD_BEGIN
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return SD_ERR_CUDA;
    const int sms = num_sms(dev);
    for (int m0 = 0; m0 < M; m0 += 8) {  // blocks of at most 8 rows of x
        const int mb = M - m0 < 8 ? M - m0 : 8;
        const cudaError_t e = launch_wb_mma(static_cast<const char*>(x) + (size_t)m0 * K * 2, tiled_qweight,
                                            tiled_sz, bits, mb, N, K, static_cast<char*>(out) + (size_t)m0 * N * 2,
                                            sms, s);
        if (e != cudaSuccess) return SD_ERR_CUDA;
    }
    return SD_OK;
    SD_GUARD_END
}

sd_status sd_a4_quantize(const void* x, int M, int K, void* qx, float* sx, void* stream) {
    SD_INJECT("sd_a4_quantize");
    if (!x || !qx || !sx) return SD_ERR_INVALID_ARG;
    if (M <= 0 || K <= 0 || K % 128 != 0) return SD_ERR_INVALID_ARG;
    if (!aligned(x, 16) || !aligned(qx, 16) || !aligned(sx, 4)) return SD_ERR_INVALID_ARG;
    SD_GUARD_BEGIN
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return SD_ERR_CUDA;
    int* err = device_error_word(dev);
    if (!err) return SD_ERR_CUDA;
    return from_cuda(launch_a4_quantize(x, M, K, qx, sx, err, num_sms(dev), static_cast<cudaStream_t>(stream)));
    SD_GUARD_END
}

sd_status sd_w4a4_linear_tiled(const void* qx, const float* sx, const void* tiled_qweight, const void* tiled_sz,
                               int group, int M, int N, int K, void* out, void* stream) {
    SD_INJECT("sd_w4a4_linear_tiled");
    if (!qx || !sx || !tiled_qweight || !tiled_sz || !out) return SD_ERR_INVALID_ARG;
    if (M <= 0 || N <= 0 || K <= 0 || group <= 0 || K % group != 0) return SD_ERR_INVALID_ARG;
    if (!aligned(qx, 16) || !aligned(sx, 4) || !aligned(tiled_qweight, 16) || !aligned(tiled_sz, 16) ||
        !aligned(out, 2))
        return SD_ERR_INVALID_ARG;
    if (group != 128) return SD_ERR_UNSUPPORTED;
    SD_GUARD_BEGIN
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return SD_ERR_CUDA;
    const int sms = num_sms(dev);
    const int G = K / 128;
    for (int m0 = 0; m0 < M; m0 += 8) {  // blocks of at most 8 rows of x
        const int mb = M - m0 < 8 ? M - m0 : 8;
        const cudaError_t e = launch_w4a4_mma(static_cast<const char*>(qx) + (size_t)m0 * K * 2, sx + (size_t)m0 * G,
                                              tiled_qweight, tiled_sz, mb, N, K,
                                              static_cast<char*>(out) + (size_t)m0 * N * 2, sms, s);
        if (e != cudaSuccess) return SD_ERR_CUDA;
    }
    return SD_OK;
    SD_GUARD_END
}

sd_status sd_w8a16_linear(const void* x, const int8_t* qweight, const void* scales, int M, int N,
                          int K, void* out, void* stream) {
    SD_INJECT("sd_w8a16_linear");
    if (!x || !qweight || !scales || !out) return SD_ERR_INVALID_ARG;
    if (M <= 0 || N <= 0 || K <= 0 || K % 16 != 0) return SD_ERR_INVALID_ARG;
    if (!aligned(x, 16) || !aligned(qweight, 16) || !aligned(scales, 2) || !aligned(out, 2))
        return SD_ERR_INVALID_ARG;
    SD_GUARD_BEGIN
    return from_cuda(launch_gemv(1, x, qweight, scales, nullptr, M, N, K, out,
                                 static_cast<cudaStream_t>(stream)));
    SD_GUARD_END
}

sd_status sd_bf16_linear(const void* x, const void* w, int M, int N, int K, void* out,
                         void* stream) {
    SD_INJECT("sd_bf16_linear");
    if (!x || !w || !out) return SD_ERR_INVALID_ARG;
    if (M <= 0 || N <= 0 || K <= 0 || K % 8 != 0) return SD_ERR_INVALID_ARG;
    if (!aligned(x, 16) || !aligned(w, 16) || !aligned(out, 2)) return SD_ERR_INVALID_ARG;
    SD_GUARD_BEGIN
    return from_cuda(launch_gemv(2, x, w, nullptr, nullptr, M, N, K, out,
                                 static_cast<cudaStream_t>(stream)));
    SD_GUARD_END
}

sd_status sd_w4_unpack(const uint32_t* qweight, int N, int K, uint8_t* q, void* stream) {
    SD_INJECT("sd_w4_unpack");
    if (!qweight || !q || N <= 0 || K <= 0 || K % 8 != 0) return SD_ERR_INVALID_ARG;
    if (!aligned(qweight, 4)) return SD_ERR_INVALID_ARG;
    SD_GUARD_BEGIN
    return from_cuda(launch_w4_unpack(qweight, N, K, q, static_cast<cudaStream_t>(stream)));
    SD_GUARD_END
}

sd_status sd_philox4x32(const uint32_t* ctr, uint32_t key0, uint32_t key1, int n, uint32_t* out,
                        void* stream) {
    SD_INJECT("sd_philox4x32");
    if (!ctr || !out || n <= 0) return SD_ERR_INVALID_ARG;
    if (!aligned(ctr, 16) || !aligned(out, 16)) return SD_ERR_INVALID_ARG;
    SD_GUARD_BEGIN
    return from_cuda(launch_philox(ctr, key0, key1, n, out, static_cast<cudaStream_t>(stream)));
    SD_GUARD_END
}

sd_status sd_verify(const float* draft_logits, const float* target_logits,
                    const int32_t* draft_tokens, int gamma, int batch, int vocab,
                    float temperature, uint64_t seed, int32_t* out_tokens,
                    int32_t* out_accept_len, void* stream) {
    SD_INJECT("sd_verify");
    if (gamma < 1 || gamma > 16 || batch < 0 || vocab < 1) return SD_ERR_INVALID_ARG;
    if (!(temperature >= 0.f) || (temperature > 0.f && temperature < 1e-6f) || temperature > 1e6f)
        return SD_ERR_INVALID_ARG;
    if (!target_logits || !draft_tokens || !out_tokens || !out_accept_len) return SD_ERR_INVALID_ARG;
    if (temperature > 0.f && !draft_logits) return SD_ERR_INVALID_ARG;
    if (!aligned(target_logits, 4) || (draft_logits && !aligned(draft_logits, 4)) ||
        !aligned(draft_tokens, 4) || !aligned(out_tokens, 4) || !aligned(out_accept_len, 4))
        return SD_ERR_INVALID_ARG;
    if (batch == 0) return SD_OK;
    SD_GUARD_BEGIN
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return SD_ERR_CUDA;
    const int sms = num_sms(dev);
    int* err = device_error_word(dev);
    if (!err) return SD_ERR_CUDA;
    const size_t need = verify_workspace_bytes(gamma, batch, vocab, temperature, sms);
    void* ws = workspace(0, dev, s, need);
    unsigned* cnt = counters(0, dev, s, verify_counter_count(batch));
    if (!ws || !cnt) return SD_ERR_CUDA;
    VerifyArgs a{draft_logits, target_logits, draft_tokens, gamma, batch, vocab,
                 temperature, seed, out_tokens, out_accept_len};
    return from_cuda(launch_verify(a, ws, need, cnt, sms, err, s));
    SD_GUARD_END
}

sd_status sd_sample(const float* logits, int batch, int vocab, float temperature, uint64_t seed,
                    int slot, int32_t* out_tokens, void* stream) {
    SD_INJECT("sd_sample");
    if (!logits || !out_tokens || batch < 0 || vocab < 1 || slot < 0 || slot > (1 << 30))
        return SD_ERR_INVALID_ARG;
    if (!(temperature >= 0.f) || (temperature > 0.f && temperature < 1e-6f) || temperature > 1e6f)
        return SD_ERR_INVALID_ARG;
    if (!aligned(logits, 4) || !aligned(out_tokens, 4)) return SD_ERR_INVALID_ARG;
    if (batch == 0) return SD_OK;
    SD_GUARD_BEGIN
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return SD_ERR_CUDA;
    const int sms = num_sms(dev);
    const size_t need = sample_workspace_bytes(batch, vocab, sms);
    void* ws = workspace(2, dev, s, need);
    unsigned* cnt = counters(2, dev, s, (size_t)batch);
    if (!ws || !cnt) return SD_ERR_CUDA;
    return from_cuda(launch_sample(logits, batch, vocab, temperature, seed, slot, out_tokens, ws, need, cnt, sms, s));
    SD_GUARD_END
}

sd_status sd_lm_head_parts(int M, int vocab, int K, int* parts) {
    SD_INJECT("sd_lm_head_parts");
    if (!parts || M < 1 || M > 32 || vocab < 1 || K < 128 || K % 128 != 0) return SD_ERR_INVALID_ARG;
    SD_GUARD_BEGIN
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return SD_ERR_CUDA;
    const int n = w4a16_lm_head_parts(M, vocab, K, num_sms(dev));
    if (n < 1) return SD_ERR_CUDA;
    *parts = n;
    return SD_OK;
    SD_GUARD_END
}

sd_status sd_w4a16_lm_head(const void* x, const void* tiled_qweight, const void* tiled_sz, int group,
                           int M, int vocab, int K, float temperature, float* logits, int64_t ld_logits,
                           void* stats, int64_t ld_stats, void* stream) {
    SD_INJECT("sd_w4a16_lm_head");
    if (!x || !tiled_qweight || !tiled_sz || !logits || !stats) return SD_ERR_INVALID_ARG;
    if (M <= 0 || vocab <= 0 || K <= 0 || group <= 0 || K % 8 != 0 || K % group != 0)
        return SD_ERR_INVALID_ARG;
    if (!(temperature >= 0.f) || (temperature > 0.f && temperature < 1e-6f) || temperature > 1e6f)
        return SD_ERR_INVALID_ARG;
    if (!aligned(x, 16) || !aligned(tiled_qweight, 16) || !aligned(tiled_sz, 16) || !aligned(logits, 4) ||
        !aligned(stats, 8))
        return SD_ERR_INVALID_ARG;
    if (ld_logits < vocab) return SD_ERR_INVALID_ARG;
    if (group != 128) return SD_ERR_UNSUPPORTED;
    if (M > 32) return SD_ERR_UNSUPPORTED;
    SD_GUARD_BEGIN
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return SD_ERR_CUDA;
    const int sms = num_sms(dev);
    const int parts = w4a16_lm_head_parts(M, vocab, K, sms);
    if (parts < 1) return SD_ERR_CUDA;
    if (ld_stats < parts) return SD_ERR_INVALID_ARG;
    return from_cuda(launch_w4a16_lm_head(x, tiled_qweight, tiled_sz, M, vocab, K, temperature, logits,
                                          (long long)ld_logits, stats, (long long)ld_stats, sms, s));
    SD_GUARD_END
}

sd_status sd_verify_parts(const float* draft_logits, const float* target_logits,
                          const void* draft_stats, int draft_parts, const void* target_stats,
                          int target_parts, const int32_t* draft_tokens, int gamma, int batch,
                          int vocab, float temperature, uint64_t seed, int32_t* out_tokens,
                          int32_t* out_accept_len, void* stream) {
    SD_INJECT("sd_verify_parts");
    if (gamma < 1 || gamma > 16 || batch < 0 || vocab < 1) return SD_ERR_INVALID_ARG;
    if (!(temperature >= 0.f) || (temperature > 0.f && temperature < 1e-6f) || temperature > 1e6f)
        return SD_ERR_INVALID_ARG;
    if (!target_logits || !target_stats || !draft_tokens || !out_tokens || !out_accept_len)
        return SD_ERR_INVALID_ARG;
    if (target_parts < 1) return SD_ERR_INVALID_ARG;
    if (temperature > 0.f && (!draft_logits || !draft_stats || draft_parts < 1)) return SD_ERR_INVALID_ARG;
    if (!aligned(target_logits, 4) || (draft_logits && !aligned(draft_logits, 4)) ||
        !aligned(target_stats, 8) || (draft_stats && !aligned(draft_stats, 8)) ||
        !aligned(draft_tokens, 4) || !aligned(out_tokens, 4) || !aligned(out_accept_len, 4))
        return SD_ERR_INVALID_ARG;
    if (batch == 0) return SD_OK;
    SD_GUARD_BEGIN
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return SD_ERR_CUDA;
    const int sms = num_sms(dev);
    int* err = device_error_word(dev);
    if (!err) return SD_ERR_CUDA;
    const int parts = temperature > 0.f && draft_parts > target_parts ? draft_parts : target_parts;
    const size_t need = verify_workspace_bytes(gamma, batch, vocab, temperature, sms, parts);
    void* ws = workspace(0, dev, s, need);
    unsigned* cnt = counters(0, dev, s, verify_counter_count(batch));
    if (!ws || !cnt) return SD_ERR_CUDA;
    VerifyArgs a{draft_logits, target_logits, draft_tokens, gamma, batch, vocab,
                 temperature, seed, out_tokens, out_accept_len};
    return from_cuda(launch_verify_parts(a, temperature > 0.f ? draft_stats : nullptr,
                                         temperature > 0.f ? draft_parts : 0, target_stats, target_parts,
                                         ws, need, cnt, sms, err, s));
    SD_GUARD_END
}

sd_status sd_verify_noalloc(const float* draft_logits, const float* target_logits,
                            const int32_t* draft_tokens, int gamma, int batch, int vocab,
                            float temperature, uint64_t seed, int32_t* out_tokens,
                            int32_t* out_accept_len, void* stream) {
    SD_INJECT("sd_verify_noalloc");
    if (gamma < 1 || gamma > 16 || batch < 0 || vocab < 1) return SD_ERR_INVALID_ARG;
    if (!(temperature >= 0.f) || (temperature > 0.f && temperature < 1e-6f) || temperature > 1e6f)
        return SD_ERR_INVALID_ARG;
    if (!target_logits || !draft_tokens || !out_tokens || !out_accept_len) return SD_ERR_INVALID_ARG;
    if (temperature > 0.f && !draft_logits) return SD_ERR_INVALID_ARG;
    if (!aligned(target_logits, 4) || (draft_logits && !aligned(draft_logits, 4)) ||
        !aligned(draft_tokens, 4) || !aligned(out_tokens, 4) || !aligned(out_accept_len, 4))
        return SD_ERR_INVALID_ARG;
    if (batch == 0) return SD_OK;
    SD_GUARD_BEGIN
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return SD_ERR_CUDA;
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
        return SD_ERR_CUDA;
    VerifyArgs a{draft_logits, target_logits, draft_tokens, gamma, batch, vocab,
                 temperature, seed, out_tokens, out_accept_len};
    return (sd_status)launch_verify_static(a, dev, sms, static_cast<cudaStream_t>(stream));
    SD_GUARD_END
}

sd_status sd_test_wait_expiry(int64_t cycles, void* stream) {
    SD_INJECT("sd_test_wait_expiry");
    if (cycles < 1 || cycles > (1ll << 40)) return SD_ERR_INVALID_ARG;
    SD_GUARD_BEGIN
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return SD_ERR_CUDA;
    int* err = device_error_word(dev);
    if (!err) return SD_ERR_CUDA;
    return from_cuda(launch_wait_expiry((long long)cycles, err, static_cast<cudaStream_t>(stream)));
    SD_GUARD_END
}

sd_status sd_device_error(void* stream, int32_t* code) {
    SD_INJECT("sd_device_error");
    if (!code) return SD_ERR_INVALID_ARG;
    SD_GUARD_BEGIN
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return SD_ERR_CUDA;
    int* err = device_error_word(dev);
    if (!err) return SD_ERR_CUDA;
    int* err2 = verify_static_error_word(dev);  // the allocation-free path's word
    int host[2] = {0, 0};
    if (cudaMemcpyAsync(&host[0], err, sizeof(int), cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return SD_ERR_CUDA;
    if (cudaMemsetAsync(err, 0, sizeof(int), s) != cudaSuccess) return SD_ERR_CUDA;
    if (err2) {
        if (cudaMemcpyAsync(&host[1], err2, sizeof(int), cudaMemcpyDeviceToHost, s) != cudaSuccess)
            return SD_ERR_CUDA;
        if (cudaMemsetAsync(err2, 0, sizeof(int), s) != cudaSuccess) return SD_ERR_CUDA;
    }
    if (cudaStreamSynchronize(s) != cudaSuccess) return SD_ERR_CUDA;
    *code = host[0] ? host[0] : host[1];
    return SD_OK;
    SD_GUARD_END
}

}  // extern "C"
