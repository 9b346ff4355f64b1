// Internal host-side declarations shared by the translation units of libsd.so.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace sd {

// Per-device error word (int, zero = no error) that kernels record
// data-dependent errors into.  Allocated on first use; never freed.
int* device_error_word(int device);

int num_sms(int device);

// CUDA-core GEMV family, M <= 8.  fmt: 0 = W4 g128, 1 = W8 per-channel, 2 = bf16.
cudaError_t launch_gemv(int fmt, const void* x, const void* w, const void* scales,
                        const void* zeros, int M, int N, int K, void* out, cudaStream_t s);

// Tensor-core (tcgen05) W4A16 GEMM, any M <= 160, group 128, K % 128 == 0.
// Its K splits meet inside a thread-block cluster: the workspace size is 0 and
// ws / counters are not used.
size_t w4a16_tc_workspace_bytes(int M, int N, int K, int sms);
cudaError_t launch_w4a16_tc(const void* x, const uint32_t* qweight, const void* scales,
                            const void* zeros, int M, int N, int K, void* out, void* ws,
                            size_t ws_bytes, unsigned* counters, int sms, int* err,
                            cudaStream_t s);

// Tensor-core W4A16 for 1 <= M <= 32: TMA weight stream, dequantisation into
// TMEM, group scaling after the MMA.  Same workspace/counter contract.
int w4a16_tc2_splits(int M, int N, int K, int sms);
size_t w4a16_tc2_workspace_bytes(int M, int N, int K, int sms);
cudaError_t launch_w4a16_tc2(const void* x, const uint32_t* qweight, const void* scales,
                             const void* zeros, int M, int N, int K, void* out, void* ws,
                             size_t ws_bytes, unsigned* counters, int sms, int* err,
                             cudaStream_t s);

// Register-operand (mma.sync) W4A16 for 1 <= M <= 32 on the fragment-ordered
// layout of sd_w4_tile: wq [ceil(N/16)][K/64][32] 16-byte units, wsz
// [ceil(N/16)][K/128][8] 8-byte entries {(s, bf16 128 + z) of row g, of row
// g + 8}.  K splits meet in distributed shared memory: no workspace.
void w4_tiled_sizes(int N, int K, size_t* q_bytes, size_t* sz_bytes);
cudaError_t launch_w4_tile(const uint32_t* qweight, const void* scales, const void* zeros, int N,
                           int K, void* wq, void* wsz, int* err, int sms, cudaStream_t s);
cudaError_t launch_w4a16_mma(const void* x, const void* wq, const void* wsz, int M, int N, int K,
                             void* out, int sms, cudaStream_t s);

// The same kernel reading the sd_w4_pack layout directly (row-major qweight,
// fp16 scales and zeros), 1 <= M <= 32; needs K % 256 == 0 (an even number of
// groups), qweight 16-byte and scales / zeros 4-byte aligned
// (w4a16_mma_rowmajor_ok).
bool w4a16_mma_rowmajor_ok(const void* qweight, const void* scales, const void* zeros, int M, int K);
cudaError_t launch_w4a16_mma_rowmajor(const void* x, const uint32_t* qweight, const void* scales, const void* zeros,
                                      int M, int N, int K, void* out, int sms, cudaStream_t s);

// The same kernel on b-bit weights (b = 2, 3; 1 <= M <= 8): wq holds, per
// 16-row tile and 128-input group, 32 lanes x 16 bytes of 2-bit pairs and, for
// b = 3, 32 lanes x 8 bytes of third bits; wsz as for INT4.  b = 4 runs the
// INT4 kernel.  wb_tile converts the row-major b-bit stream of sd_wb_pack.
void wb_tiled_sizes(int N, int K, int bits, size_t* q_bytes, size_t* sz_bytes);
cudaError_t launch_wb_tile(const uint32_t* packed, const void* scales, const void* zeros, int bits, int N,
                           int K, void* wq, void* wsz, int* err, int sms, cudaStream_t s);
cudaError_t launch_wb_mma(const void* x, const void* wq, const void* wsz, int bits, int M, int N, int K, void* out,
                          int sms, cudaStream_t s);
// W4A4 (1 <= M <= 8): activation codes as bf16 integers qx [M][K] with fp32
// scales sx [M][K/128] (launch_a4_quantize), against the tiled INT4 weights.
cudaError_t launch_a4_quantize(const void* x, int M, int K, void* qx, float* sx, int* err, int sms,
                               cudaStream_t s);
cudaError_t launch_w4a4_mma(const void* qx, const float* sx, const void* wq, const void* wsz, int M, int N, int K,
                            void* out, int sms, cudaStream_t s);

// Logits mode of the same kernel (the lm_head), 1 <= M <= 32: fp32 logits
// [M] rows of stride ld_logits, and per x row one softmax partial per CTA in
// stats [M] rows of stride ld_stats >= w4a16_lm_head_parts(M, N, K, sms):
// (max logit, sum exp((l - max) / T)) for T > 0, (max logit, argmax index as
// int bits) for T = 0.  parts is -1 for an unsupported shape.
int w4a16_lm_head_parts(int M, int N, int K, int sms);
cudaError_t launch_w4a16_lm_head(const void* x, const void* wq, const void* wsz, int M, int N, int K,
                                 float temperature, float* logits, long long ld_logits, void* stats,
                                 long long ld_stats, int sms, cudaStream_t s);

// Test kernel: one bounded mbarrier wait (the tensor-core kernels' routine)
// on a barrier nothing arrives on; records SD_ERR_TIMEOUT in err.
cudaError_t launch_wait_expiry(long long cycles, int* err, cudaStream_t s);

cudaError_t launch_w4_unpack(const uint32_t* qweight, int N, int K, uint8_t* q, cudaStream_t s);
cudaError_t launch_philox(const uint32_t* ctr, uint32_t k0, uint32_t k1, int n, uint32_t* out,
                          cudaStream_t s);

struct VerifyArgs {
    const float* draft;
    const float* target;
    const int32_t* tokens;
    int gamma, batch, vocab;
    float temperature;
    uint64_t seed;
    int32_t* out_tokens;
    int32_t* out_len;
};

// Workspace bytes the verify kernels need for a problem of this size; parts > 0:
// for launch_verify_parts with at most `parts` partials per row.
size_t verify_workspace_bytes(int gamma, int batch, int vocab, float temperature, int sms, int parts = 0);
// Number of dedicated counters the verify kernels need (zero on entry, and
// zero again when the kernels complete).
size_t verify_counter_count(int batch);
// Enqueue the verify kernels on s using ws (ws_bytes >= verify_workspace_bytes).
cudaError_t launch_verify(const VerifyArgs& a, void* ws, size_t ws_bytes, unsigned* counters,
                          int sms, int* err, cudaStream_t s);

// The same verification with the row statistics merged from lm_head partials
// (launch_w4a16_lm_head): target [batch][gamma + 1][target_parts], draft
// [batch][gamma][draft_parts] (unused at T = 0).  Same workspace and counters.
cudaError_t launch_verify_parts(const VerifyArgs& a, const void* draft_stats, int draft_parts,
                                const void* target_stats, int target_parts, void* ws, size_t ws_bytes,
                                unsigned* counters, int sms, int* err, cudaStream_t s);

// Draft-side sampler (sd_sample): workspace bytes and launch; counters: batch
// dedicated zero-initialised counters.
size_t sample_workspace_bytes(int batch, int vocab, int sms);
cudaError_t launch_sample(const float* logits, int batch, int vocab, float temperature, uint64_t seed, int slot,
                          int32_t* out, void* ws, size_t ws_bytes, unsigned* counters, int sms, cudaStream_t s);

// Allocation-free verify: scratch in a fixed 1 MiB device array; returns an
// sd_status value.  `dev` is the current device.
int launch_verify_static(const VerifyArgs& a, int dev, int sms, cudaStream_t s);
// Error word of the allocation-free path on `dev` (current device), or nullptr.
int* verify_static_error_word(int dev);

}  // namespace sd
