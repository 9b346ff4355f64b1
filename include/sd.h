/*
 * sd.h -- C ABI of the GB300 quantized speculative-decoding hot path.
 *
 * Two operations, as the pages state the problem:
 *   1. the weight-only quantized linear layer that the draft and the target
 *      run ("The Free Half of Speculative Decoding", para. 3: INT4 AWQ target
 *      and quantized draft; "When Do Quantized Drafts Help Speculative
 *      Decoding?", "Current pilot setup": BF16 / GPTQ INT8 / GPTQ INT4 draft,
 *      gamma = 4, batch 1);
 *   2. the speculative-sampling verification of gamma drafted tokens ("The
 *      Free Half ...", para. 4: the target verifies every proposed token;
 *      "When Do Quantized Drafts ...", References [2] Leviathan et al. and
 *      [3] Chen et al.: accept with probability min(1, p/q), resample the first
 *      rejected slot from norm(max(0, p - q)), bonus token from p_{gamma+1}).
 * Around them: the host weight packers (INT4, INT8, and INT2 / INT3 / INT4
 * bit streams), the draft's token draw (sd_sample), and the INT4 lm_head
 * that writes, beside its logits, the softmax partials the verification
 * merges instead of re-reading the rows (sd_w4a16_lm_head, sd_verify_parts).
 *
 * Conventions for every call:
 *   - Return value: sd_status.  Argument checks run on the host first; on
 *     failure SD_ERR_INVALID_ARG (or SD_ERR_UNSUPPORTED) is returned and
 *     nothing is launched or written.
 *   - Device calls take DEVICE pointers and a CUDA stream (a cudaStream_t
 *     passed as void*; NULL = the legacy default stream).  They enqueue work
 *     and return without synchronising; a launch failure returns
 *     SD_ERR_CUDA.  Faults inside kernels surface at the caller's next
 *     synchronisation, like any CUDA kernel.
 *   - Ownership: the caller owns every buffer passed in.  The library keeps
 *     no pointer after a call returns.
 *   - Data-dependent errors detected on the device (a draft token outside
 *     [0, vocab)) do not fault: the kernel records the code in a device
 *     error word that sd_device_error() reads and clears.
 *   - Exceptions never cross this boundary.
 *   - Kernels are launched with programmatic dependent launch: a call may
 *     start while the previous kernel on its stream is still draining, and
 *     waits for it before reading activations / logits or writing anything.
 *     The tensor-core linear calls read their packed weights, scales and
 *     zeros BEFORE that wait; those arrays must therefore be complete before
 *     the call is enqueued (e.g. synchronise after sd_w4_tile or an upload).
 *   - The environment variable SD_FAULT_INJECT="<function>:<status>[,...]"
 *     makes the named functions return <status> without doing anything
 *     (host-side fault injection for error-path tests).
 *
 * Linear-layer layout: y[M][N] = x[M][K] . W[N][K]^T (nn.Linear layout), x and
 * y row-major bf16, fp32 accumulation.
 */
#ifndef SD_H_
#define SD_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum sd_status {
    SD_OK = 0,
    SD_ERR_INVALID_ARG = 1, /* bad pointer, size or value; nothing launched */
    SD_ERR_UNSUPPORTED = 2, /* valid but not implemented (e.g. group != 128) */
    SD_ERR_CUDA = 3,        /* a CUDA runtime call or launch failed */
    SD_ERR_TIMEOUT = 4,     /* a bounded device-side wait gave up */
    SD_ERR_INTERNAL = 5     /* anything else (allocation, host exception) */
} sd_status;

/* Static string for a status code (never NULL). */
const char* sd_status_string(int status);

/* ABI version, (major << 16) | minor. */
int sd_version(void);

/* ---------------------------------------------------------------- packers
 * Host-side, synchronous, CPU only.  All pointers are HOST pointers.
 *
 * sd_w4_pack: asymmetric uint4 round-to-nearest group quantisation of fp32
 * weights w[N][K] along K with `group` consecutive inputs per group (the
 * INT4 AWQ / GPTQ weight format of "The Free Half ...", para. 3, and "When Do
 * Quantized Drafts ...", pilot setup).  Per (n, group g):
 *   lo = min(0, min w), hi = max(0, max w);
 *   s  = (hi - lo)/15 rounded to fp16 (nearest even), raised one fp16 ulp if
 *        15*s < hi - lo; s = 1 when hi == lo;
 *   z  = clamp(round_even(-lo/s), 0, 15)          (stored as an fp16 integer)
 *   q  = clamp(round_even(w/s) + z, 0, 15),   dequantised w' = (q - z) * s.
 * Outputs (caller-allocated):
 *   qweight uint32 [N][K/8]: nibble j (bits 4j..4j+3) of word (n, c) holds
 *                            q[n][8c + j];
 *   scales  fp16 bits [N][K/group];  zeros fp16 bits [N][K/group].
 * Errors: SD_ERR_INVALID_ARG for NULL pointers, N/K <= 0, K % 8 != 0,
 * group <= 0, K % group != 0, a non-finite weight, or a scale that overflows
 * fp16.
 */
sd_status sd_w4_pack(const float* w, int N, int K, int group, uint32_t* qweight,
                     uint16_t* scales, uint16_t* zeros);

/* sd_wb_pack: sd_w4_pack for b-bit weights, b = bits in {2, 3, 4} (the INT4,
 * INT3 and INT2 targets of "Speculative Decoding in Quantized Regimes",
 * sec. 4.1-4.2): the same rules with L = 2^b - 1 levels in place of 15
 * (s = (hi - lo)/L rounded to fp16 and stepped up if L*s < hi - lo;
 * z = clamp(round_even(-lo/s), 0, L); q = clamp(round_even(w/s) + z, 0, L)).
 * Output layout: each row's codes form one little-endian bit stream along K,
 * code k in bits b*k .. b*k + b - 1, stored as uint32 words
 *   packed uint32 [N][K*b/32] (word c holds stream bits 32c .. 32c + 31);
 * an INT3 code can straddle two words.  b = 4 gives sd_w4_pack's layout.
 *   scales, zeros fp16 bits [N][K/group] as sd_w4_pack.
 * Errors: as sd_w4_pack, plus K*b % 32 != 0 -> SD_ERR_INVALID_ARG; bits
 * outside {2, 3, 4} -> SD_ERR_UNSUPPORTED.  sd_wb_tile copies this layout
 * into the one sd_wb_linear_tiled reads. */
sd_status sd_wb_pack(const float* w, int N, int K, int group, int bits, uint32_t* packed,
                     uint16_t* scales, uint16_t* zeros);

/* sd_w8_pack: symmetric INT8 per-output-channel quantisation (the GPTQ INT8
 * draft of "When Do Quantized Drafts ...", pilot setup):
 *   s = max|w[n][:]|/127 rounded to fp16, raised one ulp if 127*s < max|w|,
 *       s = 1 for an all-zero row;  q8 = clamp(round_even(w/s), -127, 127).
 * Outputs: qweight int8 [N][K], scales fp16 bits [N].
 * Errors: SD_ERR_INVALID_ARG for NULL pointers, N/K <= 0, a non-finite
 * weight or an fp16 overflow of s. */
sd_status sd_w8_pack(const float* w, int N, int K, int8_t* qweight, uint16_t* scales);

/* --------------------------------------------------------- linear layers
 * sd_w4a16_linear: y = x . W'^T with W' the dequantised sd_w4_pack weights.
 *   x       bf16 [M][K] device, row-major;
 *   qweight uint32 [N][K/8] device (sd_w4_pack layout, 16-byte aligned);
 *   scales, zeros fp16 [N][K/group] device;
 *   out     bf16 [M][N] device, row-major (may not alias the inputs).
 * Arithmetic: fp32 accumulation, output rounded to bf16 (nearest even).  For
 * M <= 32 the weights enter exactly, as (q - z) * s; for M > 32 (the batched
 * tensor-core kernel) each dequantised weight (q - z) * s is computed exactly
 * in fp32 and rounded once to bf16 before the multiply.
 * Kernels: for M <= 32 with K % 256 == 0 and scales, zeros 4-byte aligned,
 * the register-operand mma.sync kernel of sd_w4a16_linear_tiled reads this
 * layout directly (no repack); other small-M cases take the CUDA-core GEMV
 * (M = 1) or the tcgen05 kernel that dequantises into tensor memory.
 * Errors: SD_ERR_INVALID_ARG for NULL pointers, M/N/K <= 0, K % 8 != 0,
 * K % group != 0, a misaligned pointer (x, qweight: 16 bytes; out, scales,
 * zeros: 2 bytes); SD_ERR_UNSUPPORTED for group != 128. */
sd_status sd_w4a16_linear(const void* x, const uint32_t* qweight, const void* scales,
                          const void* zeros, int group, int M, int N, int K, void* out,
                          void* stream);

/* sd_test_w4a16_linear_path (test hook): sd_w4a16_linear with the kernel
 * family forced, so that tests reach every kernel on every M: path 1 = the
 * CUDA-core GEMV (M <= 8; larger M -> SD_ERR_UNSUPPORTED), path 2 = the
 * tcgen05 kernels (the TMEM-dequantising kernel for M <= 32, the batched
 * kernel above), path 3 = the register-operand mma.sync kernel on the
 * row-major layout (M <= 32, K % 256 == 0, scales and zeros 4-byte aligned;
 * otherwise SD_ERR_UNSUPPORTED).  Same arithmetic, layouts and errors as
 * sd_w4a16_linear; any other path -> SD_ERR_INVALID_ARG. */
sd_status sd_test_w4a16_linear_path(const void* x, const uint32_t* qweight, const void* scales,
                                    const void* zeros, int group, int M, int N, int K, void* out, int path,
                                    void* stream);

/* ------------------------------------------------------------ tiled layout
 * A fragment-ordered copy of the sd_w4_pack weights for the small-M tensor-core
 * kernel: every 16-byte unit is what one lane of a warp feeds to four
 * mma.m16n8k16 steps, so that one warp reads 512 contiguous bytes per 16
 * output rows x 64 inputs.  With T = ceil(N/16), G = K/128:
 *   tiled_qweight: 16-byte units [T][K/64][32].  Unit (t, j, l), l = 4g + c,
 *     holds rows n_g = 16t + g and n_h = n_g + 8 at inputs k0 = 64j + 16c + 4s
 *     (s = 0..3 for its four 32-bit words, word s in bytes 4s..4s+3); the
 *     nibbles of word s, low to high, are q[n_g][k0], q[n_h][k0],
 *     q[n_g][k0+2], q[n_h][k0+2], q[n_g][k0+1], q[n_h][k0+1], q[n_g][k0+3],
 *     q[n_h][k0+3].
 *   tiled_sz: 8-byte entries [T][G][8]; entry (t, gr, g) holds two 32-bit
 *     words, for row n_g then row n_h and group gr: the fp16 scale in bits
 *     0..15 and 128 + zero as bf16 (0x4300 + z) in bits 16..31.
 *   Rows past N hold q = 0, scale 0 and zero 0.
 * The zero points must be integers in [0, 15] (sd_w4_pack writes no others).
 * Only the storage order changes: sd_w4a16_linear_tiled on the tiled copy
 * computes what sd_w4a16_linear computes on the original.
 *
 * sd_w4_tiled_bytes: the two sizes in bytes (host, no device work).  Errors:
 * NULL output pointers, N/K <= 0, K % group != 0 -> SD_ERR_INVALID_ARG;
 * group != 128 -> SD_ERR_UNSUPPORTED. */
sd_status sd_w4_tiled_bytes(int N, int K, int group, size_t* qweight_bytes, size_t* sz_bytes);

/* sd_w4_tile: builds the tiled copy on the device from the sd_w4_pack layout.
 * All pointers device; qweight, tiled_qweight and tiled_sz 16-byte aligned;
 * the caller allocates the sizes sd_w4_tiled_bytes returns.
 * Asynchronous on `stream`; a zero point that is not an integer in [0, 15]
 * is reported later as SD_ERR_INVALID_ARG by sd_device_error.
 * Errors (immediate) as sd_w4_tiled_bytes, plus NULL or misaligned pointers. */
sd_status sd_w4_tile(const uint32_t* qweight, const void* scales, const void* zeros, int group,
                     int N, int K, void* tiled_qweight, void* tiled_sz, void* stream);

/* sd_w4a16_linear_tiled: sd_w4a16_linear on the tiled copy (mma.sync kernel
 * with register-resident operands, rows of x in blocks of 32).  x and out as
 * in sd_w4a16_linear (x 16-byte aligned); tiled_qweight and tiled_sz 16-byte
 * aligned.  Arithmetic and errors as sd_w4a16_linear. */
sd_status sd_w4a16_linear_tiled(const void* x, const void* tiled_qweight, const void* tiled_sz,
                                int group, int M, int N, int K, void* out, void* stream);

/* ------------------------------------------------ INT3 / INT2 tiled layout
 * The INT4 tiled layout's idea for b-bit codes (b = 2, 3; the INT3 / INT2
 * targets of "Speculative Decoding in Quantized Regimes", sec. 4.1-4.2).  With
 * T = ceil(N/16) and G = K/128, tiled_qweight holds one block of b*256 bytes
 * per (tile t, group gr), tile-major: [T][G][b*256].  In block (t, gr), lane
 * l = 4g + c (rows n_g = 16t + g, n_h = n_g + 8) reads, for its k16 step
 * (h, s) (h = 0..1, s = 0..3), inputs k0 .. k0+3 with k0 = 128gr + 64h + 16c +
 * 4s as four code pairs i = 0..3:
 *   (n_g, k0 | k0+1), (n_h, k0 | k0+1), (n_g, k0+2 | k0+3), (n_h, k0+2 | k0+3)
 * (the INT4 layout's input order).  Bytes 16l .. 16l+15 of the block are four
 * 32-bit words; word 2h + s/2 holds the low two bits of pair i's first and
 * second code at bits 2t and 2t + 16, t = 4(s % 2) + i.  For b = 3, bytes
 * 512 + 8l .. 512 + 8l + 7 are two 32-bit words; word h holds the third bits
 * of pair i of step (h, s) at bits 4s + i and 4s + i + 16.  tiled_sz is the
 * INT4 tiled_sz (fp16 scale, bf16 128 + z per row and group).  Rows past N
 * hold code 0, scale 0 and zero 0.
 *
 * sd_wb_tiled_bytes: the two sizes in bytes (host).  bits = 4 gives the INT4
 * tiled sizes.  Errors: NULL output pointers, N/K <= 0, K % group != 0, bits
 * outside {2, 3, 4} -> SD_ERR_INVALID_ARG; group != 128 -> SD_ERR_UNSUPPORTED. */
sd_status sd_wb_tiled_bytes(int N, int K, int group, int bits, size_t* qweight_bytes, size_t* sz_bytes);

/* sd_wb_tile: builds the b-bit tiled copy on the device from sd_wb_pack's
 * stream (packed 4-byte aligned; tiled_qweight, tiled_sz 16-byte aligned;
 * scales, zeros 2-byte aligned; all device).  bits = 4 is sd_w4_tile.
 * Asynchronous; a zero point that is not an integer in [0, 2^b - 1] is
 * reported later as SD_ERR_INVALID_ARG by sd_device_error.  Errors
 * (immediate) as sd_wb_tiled_bytes, plus NULL or misaligned pointers. */
sd_status sd_wb_tile(const uint32_t* packed, const void* scales, const void* zeros, int group, int bits, int N,
                     int K, void* tiled_qweight, void* tiled_sz, void* stream);

/* sd_wb_linear_tiled: y = x . W'^T, W' = (q - z) s of the b-bit weights, on the
 * tiled copy (the mma.sync kernel of sd_w4a16_linear_tiled; rows of x in
 * blocks of 8).  x bf16 [M][K] (16-byte aligned), out bf16 [M][N]; the codes
 * enter exactly as bf16 (128 + q); fp32 accumulation, output rounded to bf16.
 * bits = 4 is sd_w4a16_linear_tiled.  Errors as sd_w4a16_linear_tiled, plus
 * bits outside {2, 3, 4} -> SD_ERR_INVALID_ARG. */
sd_status sd_wb_linear_tiled(const void* x, const void* tiled_qweight, const void* tiled_sz, int group, int bits,
                             int M, int N, int K, void* out, void* stream);

/* ------------------------------------------------------------------ W4A4
 * The W4A4 draft linear of QSPEC (cited by "When Do Quantized Drafts Help
 * Speculative Decoding?"): 4-bit activations against the shared INT4 weights.
 *
 * sd_a4_quantize: per row m and 128-input group g of x (bf16 [M][K], device,
 * 16-byte aligned; K % 128 == 0):
 *   s = fl32(max|x| / 7) (s = 1 for an all-zero group),
 *   q = clamp(round_even(fl32(x / s)), -8, 7),
 * both divisions IEEE fp32 round-to-nearest.  Outputs (device): qx bf16
 * [M][K] holding the integer codes (16-byte aligned), sx fp32 [M][K/128].
 * A non-finite input is reported later as SD_ERR_INVALID_ARG by
 * sd_device_error.  Errors (immediate): NULL or misaligned pointers, M <= 0,
 * K <= 0 or K % 128 != 0 -> SD_ERR_INVALID_ARG. */
sd_status sd_a4_quantize(const void* x, int M, int K, void* qx, float* sx, void* stream);

/* sd_w4a4_linear_tiled: y[m][n] = sum_g sx[m][g] s[n][g] sum_{k in g}
 * qx[m][k] (q[n][k] - z[n][g]) on the INT4 tiled copy.  Each group's integer
 * sum is formed exactly; fp32 accumulation over groups, output bf16 [M][N]
 * (nearest even).  qx, sx as sd_a4_quantize writes them; rows of x in blocks
 * of 8.  Errors as sd_w4a16_linear_tiled. */
sd_status sd_w4a4_linear_tiled(const void* qx, const float* sx, const void* tiled_qweight, const void* tiled_sz,
                               int group, int M, int N, int K, void* out, void* stream);

/* sd_w8a16_linear: y = x . (q8 * s)^T, INT8 per-channel weights of sd_w8_pack.
 *   x bf16 [M][K], qweight int8 [N][K] (16-byte aligned), scales fp16 [N],
 *   out bf16 [M][N]; all device.  K % 16 == 0 required.
 * Errors as sd_w4a16_linear. */
sd_status sd_w8a16_linear(const void* x, const int8_t* qweight, const void* scales, int M,
                          int N, int K, void* out, void* stream);

/* sd_bf16_linear: y = x . W^T with dense bf16 W [N][K] (the BF16 draft of "When
 * Do Quantized Drafts ...").  K % 8 == 0, W 16-byte aligned.  All device. */
sd_status sd_bf16_linear(const void* x, const void* w, int M, int N, int K, void* out,
                         void* stream);

/* sd_w4_unpack (test hook): q[n][k] = nibble of the packed layout, uint8
 * [N][K] device.  Bit-exact by definition.  K % 8 == 0. */
sd_status sd_w4_unpack(const uint32_t* qweight, int N, int K, uint8_t* q, void* stream);

/* ---------------------------------------------------------- verification
 * sd_verify: speculative-sampling verification of `gamma` drafted tokens per
 * batch element ("The Free Half ...", para. 4; "When Do Quantized Drafts
 * ...", References [2], [3]).
 *   draft_logits  fp32 [batch][gamma][vocab]      device, row-major
 *   target_logits fp32 [batch][gamma+1][vocab]    device, row-major
 *   draft_tokens  int32 [batch][gamma]            device, in [0, vocab)
 *   out_tokens    int32 [batch][gamma+1]          device: accepted draft
 *                 tokens, then the new token, then -1 padding
 *   out_accept_len int32 [batch]                  device: accepted count
 * temperature T > 0: p_i = softmax(target_i / T), q_i = softmax(draft_i / T);
 *   position i is accepted iff u_i * q_i(x_i) < p_i(x_i), u_i a Philox4x32-10
 *   uniform in [0,1) (counter (i, b, 0, 0), key = seed, word 0, top 24 bits);
 *   accept_len = first rejected position (or gamma).  The new token is drawn
 *   by an exponential race over r = max(0, p_j - q_j) at the first rejected
 *   position j (over p_j if r is all zero), or over p_gamma when all gamma
 *   are accepted: argmax_v r_v / E_v, E_v = -ln(1 - t_v),
 *   t_v = (w + 1/2) 2^-32, w = word v&3 of Philox((v>>2, b, 1+j, 0), seed).
 * temperature T == 0: greedy; position i is accepted iff x_i equals the
 *   argmax of target row i (lowest index on ties); the new token is the
 *   argmax of row accept_len.  draft_logits is not read (may be NULL).
 * Logits must be finite or -inf, with at least one finite value per row.
 * draft_logits and target_logits must be 4-byte aligned.
 * Workspace: the library allocates a small per-(device, stream) workspace on
 * the first call on a stream and keeps it for later calls; make one call per
 * stream before capturing that stream into a CUDA graph.  Calls on one stream
 * are ordered; calls on different streams use different workspaces.
 * Errors: SD_ERR_INVALID_ARG for NULL pointers, gamma outside [1, 16],
 * batch < 0, vocab < 1, T < 0, NaN, or 0 < T < 1e-6 or T > 1e6.
 * batch == 0 is a no-op.  A draft token outside [0, vocab) is treated as
 * rejected and records SD_ERR_INVALID_ARG in the device error word. */
sd_status sd_verify(const float* draft_logits, const float* target_logits,
                    const int32_t* draft_tokens, int gamma, int batch, int vocab,
                    float temperature, uint64_t seed, int32_t* out_tokens,
                    int32_t* out_accept_len, void* stream);

/* sd_verify_noalloc: sd_verify for callers that cannot allocate device memory
 * -- code that runs where cudaMalloc is not allowed or not wanted (inside an
 * engine that owns all device memory, a real-time loop that must not block on
 * the allocator, or a memory-capped sandbox).  It has no counterpart in the
 * pages; the operation, arguments, outputs and errors are those of
 * sd_verify, and the results are identical to sd_verify's.
 * Its scratch lives in a fixed 1 MiB array of device memory that the library
 * declares; every GPU that loads the library holds that array until the
 * process exits.  The call itself allocates nothing (no cudaMalloc, no
 * cudaFree, no allocating library routine) and clears the part of the array
 * that must start at zero on every call.
 * The first call on a device looks up the array's device address on that
 * device; make that first call before capturing a stream on the device.
 * All calls on a device share the one array: calls that may overlap on the
 * GPU (other streams, other threads) race and must be serialised by the
 * caller.
 * Limit: the scratch must fit in 1 MiB, about 320 bytes per batch element at
 * gamma = 16 (batch up to about 3000); a larger problem returns
 * SD_ERR_INVALID_ARG without launching anything.  Device-side errors (a draft
 * token outside [0, vocab)) are reported by sd_device_error like sd_verify's. */
sd_status sd_verify_noalloc(const float* draft_logits, const float* target_logits,
                            const int32_t* draft_tokens, int gamma, int batch, int vocab,
                            float temperature, uint64_t seed, int32_t* out_tokens,
                            int32_t* out_accept_len, void* stream);

/* sd_sample: the draft model's token draw for one draft position ("When Do
 * Quantized Drafts Help Speculative Decoding?", pilot setup: the draft proposes
 * gamma tokens, x_i ~ q_i; References [2], [3]).  For every row b:
 *   T > 0:  out_tokens[b] = argmax_v p_v / E_v, p = softmax(logits_b / T),
 *           E_v = -ln(1 - t_v), t_v = (w + 1/2) 2^-32, w = word v&3 of
 *           Philox4x32-10((v>>2, b, 1 + slot, 1), seed) -- an exact draw
 *           from p (exponential race); the lowest v wins equal keys.  The
 *           fourth counter word 1 keeps these draws apart from sd_verify's.
 *   T == 0: the argmax of the row, lowest index on ties.
 *   logits      fp32 [batch][vocab] device, row-major, 4-byte aligned;
 *               finite or -inf, at least one finite value per row;
 *   slot        the draft position (0 .. 2^30), one independent stream each;
 *   out_tokens  int32 [batch] device.
 * Workspace: as sd_verify (per device and stream, kept across calls).
 * Errors: SD_ERR_INVALID_ARG for NULL or misaligned pointers, batch < 0,
 * vocab < 1, slot < 0 or > 2^30, T < 0, NaN, 0 < T < 1e-6 or T > 1e6;
 * batch == 0 is a no-op. */
sd_status sd_sample(const float* logits, int batch, int vocab, float temperature, uint64_t seed,
                    int slot, int32_t* out_tokens, void* stream);

/* ------------------------------------- lm_head fused with the statistics
 * The target's lm_head produces the logits the verification reads ("When Do
 * Quantized Drafts ...", pilot setup; the rule of References [2], [3]
 * normalises every row by its softmax).  sd_w4a16_lm_head writes, beside the
 * fp32 logits, a set of softmax partials per row, one per CTA of its launch.
 * sd_verify_parts merges those partials instead of passing over the rows: of
 * the logits it reads only the entries at the draft tokens and the one or
 * two rows of the race.
 *
 * sd_lm_head_parts: *parts = how many partials per row sd_w4a16_lm_head
 * writes for (M, vocab, K) on the current device.  Host query; the same for
 * every call with the same arguments on the same device.
 * Errors: NULL parts, M outside [1, 32], vocab < 1, K < 128 or
 * K % 128 != 0 -> SD_ERR_INVALID_ARG; SD_ERR_CUDA if no device answers. */
sd_status sd_lm_head_parts(int M, int vocab, int K, int* parts);

/* sd_w4a16_lm_head: logits = x . W'^T for an INT4 lm_head W' [vocab][K]
 * (the tiled copy from sd_w4_tile), M <= 32 rows of x, written as fp32 (the
 * verification's input type), plus the rows' softmax partials.
 *   x       bf16 [M][K] device, 16-byte aligned;
 *   logits  fp32 device; row m starts at logits + m * ld_logits
 *           (ld_logits >= vocab); 4-byte aligned;
 *   stats   device pairs of fp32; row m starts at pair m * ld_stats
 *           (ld_stats >= sd_lm_head_parts(M, vocab, K)); 8-byte aligned.
 *           Pair i of row m covers the logits of row m that CTA i stored:
 *           T > 0:  (a, s) = (their max, sum of exp((l - a) / T));
 *           T == 0: (their max, the lowest index holding it, as int32 bits).
 *           A CTA that stored none writes (-inf, 0) or (-inf, INT32_MAX).
 * The logits' arithmetic is that of sd_w4a16_linear at M <= 32 (exact
 * dequantisation, fp32 accumulation), without the bf16 rounding.
 * The strides let draft step i fill row (b, i) of [batch][gamma][vocab]
 * logits and [batch][gamma][parts] partials: logits + i * vocab with
 * ld_logits = gamma * vocab, stats + 2 * i * parts floats with
 * ld_stats = gamma * parts.
 * Errors: as sd_w4a16_linear_tiled; M > 32 -> SD_ERR_UNSUPPORTED; NULL
 * logits or stats, ld_logits < vocab, ld_stats < parts, misaligned logits
 * or stats, T < 0, NaN, 0 < T < 1e-6 or T > 1e6 -> SD_ERR_INVALID_ARG. */
sd_status sd_w4a16_lm_head(const void* x, const void* tiled_qweight, const void* tiled_sz, int group,
                           int M, int vocab, int K, float temperature, float* logits, int64_t ld_logits,
                           void* stats, int64_t ld_stats, void* stream);

/* sd_verify_parts: sd_verify with the rows' softmax statistics merged from
 * sd_w4a16_lm_head partials taken at the same temperature.
 *   target_stats [batch][gamma+1][target_parts] pairs: rows b (gamma+1) + i
 *                of one sd_w4a16_lm_head call with M = batch (gamma+1) and
 *                ld_stats = target_parts;
 *   draft_stats  [batch][gamma][draft_parts] pairs (T > 0; not read and may
 *                be NULL at T == 0).
 * Everything else (arguments, outputs, workspace, errors) as sd_verify; also
 * SD_ERR_INVALID_ARG for target_parts < 1, draft_parts < 1 at T > 0, or a
 * stats pointer that is NULL (when read) or not 8-byte aligned.  The
 * decisions equal sd_verify's on the same logits except where the fp32
 * rounding of the merged statistics decides a near tie. */
sd_status sd_verify_parts(const float* draft_logits, const float* target_logits,
                          const void* draft_stats, int draft_parts, const void* target_stats,
                          int target_parts, const int32_t* draft_tokens, int gamma, int batch,
                          int vocab, float temperature, uint64_t seed, int32_t* out_tokens,
                          int32_t* out_accept_len, void* stream);

/* sd_philox4x32 (test hook): out[i][0..3] = Philox4x32-10 of counter
 * ctr[i][0..3] under key (key0, key1) (Salmon et al., SC'11, the generator
 * the verification uniforms come from).  ctr, out: uint32 [n][4] device. */
sd_status sd_philox4x32(const uint32_t* ctr, uint32_t key0, uint32_t key1, int n,
                        uint32_t* out, void* stream);

/* sd_test_wait_expiry (test hook for the bounded device waits,
 * SD_ERR_TIMEOUT in the status list above): launches one CTA that waits on an
 * mbarrier that nothing ever arrives on, with the bounded wait routine of the
 * tensor-core W4A16 kernels' pipelines and a limit of `cycles` SM clock
 * cycles (those kernels use about 2^31, about 1 s).  No copy or MMA is in
 * flight.  The wait gives up, records SD_ERR_TIMEOUT in the device error word
 * (read it with sd_device_error) and the kernel returns, leaving the context
 * usable.  Errors: cycles < 1 or > 2^40 -> SD_ERR_INVALID_ARG. */
sd_status sd_test_wait_expiry(int64_t cycles, void* stream);

/* sd_device_error: synchronises `stream`, then returns in *code the first
 * error recorded by a kernel on this device since the last call (SD_OK if
 * none) and clears it. */
sd_status sd_device_error(void* stream, int32_t* code);

#ifdef __cplusplus
}
#endif

#endif /* SD_H_ */
