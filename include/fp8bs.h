/*
 * fp8bs -- fine-grained FP8 quantization and block-scaled FP8 GEMM for B300
 * (sm_103a).  Plain C ABI: device pointers, sizes and a CUDA stream passed as
 * an opaque pointer.  No call allocates memory.
 *
 * What the operations compute comes from the FP8 mixed-precision training
 * scheme described on the pages (a DeepSeek-V3-style framework):
 *   - "Should Fixing Deepseek Take 60 Steps?", Figure 7 (a) passage: activations
 *     are grouped and scaled per 1x128 tile (one token, 128 channels); weights
 *     per 128x128 block (128 input channels x 128 output channels).
 *   - same page, max-abs scaling passage: each group is aligned to the FP8 range
 *     by mapping its largest magnitude onto the largest FP8 value; the max-abs
 *     is taken online per tile / block (page at why-be.why-be.co.kr, online
 *     amax passage).
 *   - untitled page at jp-study.kr, hybrid-format passage: E4M3 on all tensors.
 *   - "Should Fixing Deepseek Take 60 Steps?", Figure 6 passage: Fprop, Dgrad and
 *     Wgrad run in FP8, take FP8 inputs and produce BF16 or FP32.
 *   - untitled page at jp-study.kr, Figure 7 (b) passage: partial results are
 *     promoted to FP32 registers on CUDA cores, where the scales are applied.
 *
 * Quantization (bit-exact contract, all three granularities):
 *   amax = max |x| over the tile (x widened to fp32 exactly);
 *   r    = fl32(448 / amax);  if r is not finite (amax == 0, or amax below
 *          448/FLT_MAX) the tile is treated as all-zero: s = r = 1;
 *   s    = fl32(amax / 448)   (the stored scale; x ~= dec(q) * s);
 *   q    = E4M3(fl32(x * r)), round to nearest even, finite overflow saturates
 *          to +-448, the sign of zero is kept.
 *   Codes are OCP E4M3FN bytes (bias 7, 0x7E = 448, 0x7F = NaN).
 *   NaN / Inf inputs are outside the contract.
 *
 * GEMM (promotion interval = one 128-deep K-slab):
 *   C[i][j] = sum_kb ( sum_{k in slab kb} dec(A[i][k]) * dec(B[j][k]) )
 *             * sa[kb][i] * sb(kb, j)
 *   Each slab's partial sum is produced by the tensor cores in FP32 and added
 *   into FP32 accumulators on CUDA cores with the two scales applied.
 *
 * Error behaviour: every call checks its arguments on the host before any
 * launch and returns a status; nothing is launched on error.  Launch failures
 * return FP8BS_ERR_CUDA.  Kernels never trap: a device-side wait that runs past
 * its limit, or invalid device-resident group offsets, is recorded in a device
 * error word that fp8bs_sync_status() reports and clears.  All calls are
 * asynchronous on the given stream (NULL = legacy default stream).
 *
 * Layout conventions: matrices are row-major; "ld" arguments are leading
 * dimensions in elements of that matrix's type (bytes for E4M3 codes).
 */
#ifndef FP8BS_H
#define FP8BS_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum fp8bs_status {
  FP8BS_OK = 0,
  FP8BS_ERR_INVALID_ARG = 1,     /* null pointer, negative size, ld too small */
  FP8BS_ERR_MISALIGNED = 2,      /* pointer / leading dimension alignment */
  FP8BS_ERR_UNSUPPORTED = 3,     /* shape outside the supported set (e.g. K % 128) */
  FP8BS_ERR_CUDA = 4,            /* CUDA runtime / launch error */
  FP8BS_ERR_DEVICE_TIMEOUT = 5,  /* a kernel gave up on a device-side wait */
  FP8BS_ERR_DEVICE_BAD_OFFSETS = 6, /* grouped GEMM offsets failed device validation */
  FP8BS_ERR_DEVICE_BAD_ROUTING = 7  /* dispatch: an expert id outside [0, E) */
} fp8bs_status;

typedef enum fp8bs_dtype { FP8BS_F32 = 0, FP8BS_BF16 = 1 } fp8bs_dtype;

/* Layout of the B-operand scales of fp8bs_gemm / fp8bs_grouped_gemm.
 *   BLOCK_NK: sb[(n/128)*ldsb + k/128]  one scale per 128x128 block, ldsb >= K/128
 *   BLOCK_KN: sb[(k/128)*ldsb + n/128]  one scale per 128x128 block, ldsb >= N/128
 *   PERCOL  : sb[(k/128)*ldsb + n]      one scale per column per 128-deep slab
 *                                       (128x1 tiles along K), ldsb >= N        */
typedef enum fp8bs_bscale {
  FP8BS_SB_BLOCK_NK = 0,
  FP8BS_SB_BLOCK_KN = 1,
  FP8BS_SB_PERCOL = 2
} fp8bs_bscale;

/* 1x128 activation quantizer (one scale per token per 128 channels).
 *   x  [M x K] fp32 or bf16 (xt), row stride ldx >= K elements.
 *   q  [M x K] E4M3 codes, row stride ldq >= K bytes.
 *   s  [K/128][lds] fp32, s[kb*lds + m], lds >= M (M-contiguous: the layout the
 *      GEMM reads for its A operand).
 * Requirements: K % 128 == 0 (UNSUPPORTED); x, q 16-byte aligned and
 * ldx*sizeof(xt), ldq multiples of 16 (MISALIGNED); s 4-byte aligned.
 * M == 0 or K == 0 is a no-op.  Caller owns all buffers. */
fp8bs_status fp8bs_quant_act_1x128(const void* x, fp8bs_dtype xt, int64_t M, int64_t K,
                                   int64_t ldx, uint8_t* q, int64_t ldq, float* s,
                                   int64_t lds, void* stream);

/* 128x1 activation quantizer (one scale per channel per 128 tokens), output
 * transposed so that tokens are contiguous: the K-major operand layout of the
 * Wgrad GEMM (contraction over tokens).
 *   x  [T x C] fp32 or bf16, row stride ldx >= C.
 *   qT [C x T] E4M3 codes, qT[c*ldq + t], ldq >= T.
 *   s  [T/128][lds] fp32, s[tb*lds + c], lds >= C.
 * Requirements: T % 128 == 0, C % 16 == 0 (UNSUPPORTED); x, qT 16-byte aligned,
 * ldx*sizeof(xt) and ldq multiples of 16 (MISALIGNED).
 * The codes equal those of fp8bs_quant_act_1x128 applied to x transposed. */
fp8bs_status fp8bs_quant_act_128x1(const void* x, fp8bs_dtype xt, int64_t T, int64_t C,
                                   int64_t ldx, uint8_t* qT, int64_t ldq, float* s,
                                   int64_t lds, void* stream);

/* Both activation quantizers in one pass over x (the backward pass needs the
 * 1x128 codes for Dgrad's A operand and the 128x1 codes for Wgrad, and the
 * pages keep activations in FP8 for it): x is read once and
 *   q, s    receive exactly what fp8bs_quant_act_1x128(x, ...) writes
 *           (q [T x C] row-major, ldq >= C; s[cb*lds + t], lds >= T);
 *   qT, sT  receive exactly what fp8bs_quant_act_128x1(x, ...) writes
 *           (qT [C x T], ldqT >= T; sT[tb*ldsT + c], ldsT >= C).
 * Source: "Should Fixing Deepseek Take 60 Steps?", Figure 6 and Figure 7 (a)
 * passages; untitled page at jp-study.kr, Figure 6 passage (FP8 activations
 * cached for the backward pass).
 * Requirements: T % 128 == 0 and C % 128 == 0 (UNSUPPORTED); x, q, qT 16-byte
 * aligned, ldx*sizeof(xt), ldq, ldqT multiples of 16; s, sT 4-byte aligned
 * (MISALIGNED).  T == 0 or C == 0 is a no-op. */
fp8bs_status fp8bs_quant_act_dual(const void* x, fp8bs_dtype xt, int64_t T, int64_t C,
                                  int64_t ldx, uint8_t* q, int64_t ldq, float* s, int64_t lds,
                                  uint8_t* qT, int64_t ldqT, float* sT, int64_t ldsT,
                                  void* stream);

/* Quantize-then-dispatch for MoE layers: activations quantized 1x128 directly
 * into expert-grouped rows, the A operand of fp8bs_grouped_gemm (untitled page
 * at jp-study.kr, MoE passage: activations are quantized to FP8 before the
 * up-projection and dispatched in FP8).
 *   x       [T x K] fp32 or bf16 (row stride ldx), one row per token;
 *   expert  [T] device int32, the expert of each token, in [0, E);
 *   outputs (device, caller-owned):
 *     offsets   [E+1]: expert e owns rows offsets[e] .. offsets[e+1]-1; its
 *               token count is padded to a multiple of 128;
 *     counts    [E]: tokens per expert (before padding);
 *     q, s      rows as fp8bs_quant_act_1x128 would write for the rows
 *               x[token] (q [M_cap x K], ldq; s[kb*lds + row], lds >= M_cap);
 *               within an expert, tokens in increasing token order; padding
 *               rows get codes 0 and scale 1 (a quantized zero row);
 *     token_row [T]: the row of each token;  row_token [M_cap]: the token of
 *               each row, -1 on padding rows.
 *   Rows of q and s at or past offsets[E] are left untouched.  row_token's
 *   first ceil(T / 1024) * E entries serve as scratch between the launches,
 *   so its entries at or past offsets[E] are unspecified on return.
 * Requirements: 1 <= E <= 256, K > 0, K % 128 == 0, M_cap % 128 == 0 and
 * ceil(T / 1024) * E <= 51200 (UNSUPPORTED); M_cap >= T + 127 * E, the
 * worst-case padded size (INVALID_ARG); x, q 16-byte aligned, ldx*sizeof(xt)
 * and ldq multiples of 16 (MISALIGNED).  An expert id outside [0, E) drops
 * that token (token_row -1) and is reported by fp8bs_sync_status as
 * FP8BS_ERR_DEVICE_BAD_ROUTING.  Three launches on the stream: ranks per
 * 1024-token chunk, the plan of rows and offsets, and the quantization with
 * both row maps and the padding rows. */
fp8bs_status fp8bs_quant_dispatch(const void* x, fp8bs_dtype xt, int64_t T, int64_t K,
                                  int64_t ldx, const int32_t* expert, int32_t E, uint8_t* q,
                                  int64_t ldq, float* s, int64_t lds, int64_t M_cap,
                                  int32_t* offsets, int32_t* counts, int32_t* token_row,
                                  int32_t* row_token, void* stream);

/* 128x128 weight quantizer (one scale per 128 x 128 block).
 *   w  [R x C] fp32 or bf16, row stride ldw >= C.
 *   q  [R x C] E4M3 codes (ldq >= C) -- may be NULL;
 *   qT [C x R] the same codes transposed (ldqT >= R) -- may be NULL; not both.
 *   s  [R/128][lds] fp32, s[rb*lds + cb], lds >= C/128.
 * With a weight stored as W [K_in x N_out]: qT is the B operand of Fprop
 * (rows N_out, K-major over K_in, scales BLOCK_KN) and q is the B operand of
 * Dgrad (rows K_in, K-major over N_out, scales BLOCK_NK).
 * Requirements: R % 128 == 0 and C % 128 == 0 (UNSUPPORTED); w, q, qT 16-byte
 * aligned, leading dimensions multiples of 16 bytes (MISALIGNED). */
fp8bs_status fp8bs_quant_w_128x128(const void* w, fp8bs_dtype wt, int64_t R, int64_t C,
                                   int64_t ldw, uint8_t* q, int64_t ldq, uint8_t* qT,
                                   int64_t ldqT, float* s, int64_t lds, void* stream);

/* Block-scaled FP8 GEMM  C[M x N] = A[M x K] * B[N x K]^T  (both K-major).
 *   A  E4M3 codes, row stride lda >= K bytes; sa[kb*ldsa + i] fp32, ldsa >= M
 *      (the layout fp8bs_quant_act_1x128 / _128x1 write).
 *   B  E4M3 codes, row stride ldb >= K bytes; sb in layout sb_mode (above).
 *   C  [M x N] fp32 or bf16 (ct), row stride ldc >= N; bf16 is rounded to
 *      nearest even from the FP32 accumulator.
 * Fprop  : A = Xq (1x128), B = WqT, sb = Sw as BLOCK_KN, C bf16.
 * Dgrad  : A = dYq (1x128), B = Wq, sb = Sw as BLOCK_NK, C bf16.
 * Wgrad  : A = XqT (128x1), B = dYqT (128x1), sb = S_dY as PERCOL, C fp32.
 * Requirements: K % 128 == 0; N % 128 == 0 for BLOCK modes, N % 16 == 0 for
 * PERCOL (UNSUPPORTED); A, B, C 16-byte aligned; lda, ldb, ldc*sizeof(ct)
 * multiples of 16 (MISALIGNED); sa, sb 4-byte aligned.  M, N == 0: no-op;
 * K == 0 writes zeros.  Any M >= 1 is allowed (the last row tile is ragged).
 * Each output is the FP32 sum over the 128-deep K slabs of (slab partial x sa
 * x sb); the slab order is fixed per output tile by the shape and the device's
 * number of SM pairs (forward, or last to first on every other wave of the
 * persistent walk when a wave's operand panels exceed half of L2), so repeated
 * calls give identical bits. */
fp8bs_status fp8bs_gemm(int64_t M, int64_t N, int64_t K,
                        const uint8_t* A, int64_t lda, const float* sa, int64_t ldsa,
                        const uint8_t* B, int64_t ldb, const float* sb, fp8bs_bscale sb_mode,
                        int64_t ldsb, void* C, fp8bs_dtype ct, int64_t ldc, void* stream);

/* Bytes of workspace fp8bs_gemm_ws can use for an M x N x K GEMM on the
 * current device (0: this shape runs no split).  The dense GEMM walks its
 * 256 x 256 output tiles persistently over the device's CTA pairs; when the
 * last wave is partial, its tiles can be split along K over the idle pairs,
 * each K-range leaving a 256 x 256 FP32 partial in the workspace.
 * Requirements: bytes non-NULL (INVALID_ARG); K % 128 == 0 (UNSUPPORTED). */
fp8bs_status fp8bs_gemm_workspace_size(int64_t M, int64_t N, int64_t K, size_t* bytes);

/* fp8bs_gemm with a device workspace for the split of the last wave (above):
 * the partials go to the workspace and a second kernel on the same stream adds
 * them in K order (deterministic: repeated calls give identical bits) and
 * writes C.  The tail tiles are summed in a different order than in
 * fp8bs_gemm, so the two agree within the GEMM tolerance, not bit for bit.
 *   workspace        device memory owned by the caller, 256-byte aligned
 *                    (MISALIGNED otherwise), or NULL (no split);
 *   workspace_bytes  its size; fewer K-ranges are used when it holds less than
 *                    fp8bs_gemm_workspace_size, and no split below two.
 * The workspace is written before it is read; its contents afterwards are
 * undefined.  Calls that share a workspace must be ordered (one stream).
 * All other arguments, requirements and errors are those of fp8bs_gemm. */
fp8bs_status fp8bs_gemm_ws(int64_t M, int64_t N, int64_t K,
                           const uint8_t* A, int64_t lda, const float* sa, int64_t ldsa,
                           const uint8_t* B, int64_t ldb, const float* sb, fp8bs_bscale sb_mode,
                           int64_t ldsb, void* C, fp8bs_dtype ct, int64_t ldc, void* workspace,
                           size_t workspace_bytes, void* stream);

/* Accumulating GEMM for FP32 gradients:  C[M x N] += A[M x K] * B[N x K]^T,
 * C fp32 (the Wgrad of several micro-batches summed into one FP32 gradient;
 * the pages keep gradients in FP32: untitled page at jp-study.kr, FP32 master
 * weights and gradients passage).  Each output element receives the block-
 * scaled product computed as in fp8bs_gemm, added once to its previous value
 * (whole tiles: TMA reduce-add in L2; tiles of a split last wave: by the
 * partial-sum kernel).  workspace / workspace_bytes as in fp8bs_gemm_ws
 * (NULL: no split).  K == 0 leaves C unchanged.  Other arguments,
 * requirements and errors are those of fp8bs_gemm with ct = FP8BS_F32. */
fp8bs_status fp8bs_gemm_accumulate(int64_t M, int64_t N, int64_t K,
                                   const uint8_t* A, int64_t lda, const float* sa, int64_t ldsa,
                                   const uint8_t* B, int64_t ldb, const float* sb,
                                   fp8bs_bscale sb_mode, int64_t ldsb, float* C, int64_t ldc,
                                   void* workspace, size_t workspace_bytes, void* stream);

/* fp8bs_gemm_ws for callers that cannot allocate device memory: some cannot
 * call cudaMalloc at all where they run (e.g. code that may not synchronize
 * the device or bypass the memory pool of the framework around it), and some
 * hold only their operand buffers and have no workspace to lend.  This entry
 * point allocates nothing: the K split's FP32 partials go to a 20 MiB array in
 * the library's own device memory, which every GPU that loads the library
 * holds until the process exits.  The paper has no counterpart of this call.
 *   Arguments, requirements and results are those of fp8bs_gemm_ws with a
 *   20 MiB workspace (the split is chosen the same way, so the two give
 *   bit-identical outputs).  The arguments are checked on the host first, as
 *   fp8bs_gemm_ws checks them: a bad call returns the same status and touches
 *   no device state.
 *   A shape whose fp8bs_gemm_workspace_size exceeds 20 MiB is rejected with
 *   FP8BS_ERR_UNSUPPORTED before any launch (on a 148-SM B300 no shape needs
 *   more than 74 partial tiles, 18.5 MiB).
 *   The first call on a device looks up the array's device address (the
 *   device must be current); make that first call before any stream capture.
 *   Every call uses the same array and it keeps the last call's partials; a
 *   call writes every partial it reads, so nothing needs clearing.  Calls that
 *   overlap on the GPU (other streams, other host threads) race on the array:
 *   order them on one stream. */
fp8bs_status fp8bs_gemm_static_ws(int64_t M, int64_t N, int64_t K,
                                  const uint8_t* A, int64_t lda, const float* sa, int64_t ldsa,
                                  const uint8_t* B, int64_t ldb, const float* sb,
                                  fp8bs_bscale sb_mode, int64_t ldsb, void* C, fp8bs_dtype ct,
                                  int64_t ldc, void* stream);

/* Grouped block-scaled FP8 GEMM for MoE experts: expert e owns rows
 * offsets[e] .. offsets[e+1]-1 of A and C and multiplies them by B[e]:
 *   C[i][:] = A[i][:] * B[e]^T with the scales sa (rows) and sb + e*sb_estride.
 *   offsets  DEVICE array of E+1 int32: offsets[0] == 0, non-decreasing,
 *            multiples of 128, offsets[E] <= M_cap.  Validated on the device;
 *            a violation writes nothing and is reported by fp8bs_sync_status()
 *            as FP8BS_ERR_DEVICE_BAD_OFFSETS.  Empty experts are allowed.
 *   A [M_cap x K] (lda), sa[kb*ldsa + i] (ldsa >= M_cap);
 *   B [E][N][ldb] codes, expert stride N*ldb bytes;
 *   sb per expert in layout sb_mode with stride ldsb, experts sb_estride apart;
 *   C [M_cap x N] (ldc); rows at or past offsets[E] are left untouched.
 * Requirements: 1 <= E <= 1024, M_cap % 128 == 0, plus those of fp8bs_gemm. */
fp8bs_status fp8bs_grouped_gemm(int32_t E, const int32_t* offsets, int64_t M_cap, int64_t N,
                                int64_t K, const uint8_t* A, int64_t lda, const float* sa,
                                int64_t ldsa, const uint8_t* B, int64_t ldb, const float* sb,
                                fp8bs_bscale sb_mode, int64_t ldsb, int64_t sb_estride,
                                void* C, fp8bs_dtype ct, int64_t ldc, void* stream);

/* MX (microscaling) quantizer: 1x32 groups along K with power-of-two scales
 * ("Should Fixing Deepseek Take 60 Steps?", Figure 7 (a) passage, and the page
 * at why-be.why-be.co.kr, accumulation-precision passage: both point to
 * microscaling, with the group scales applied inside the tensor cores, as the
 * next step after 1x128 / 128x128 scaling).
 *   x   [R x K] fp32 or bf16, row stride ldx elements (device);
 *   q   [R x K] E4M3 codes, row stride ldq bytes (device, caller-owned);
 *   sf  exponent words (device, caller-owned): for row r and 128-wide K block
 *       kb, sf[kb*ldsf + r] holds the UE8M0 exponents (e + 127) of the groups
 *       4kb .. 4kb+3 of that row in bytes 0..3.
 * A group with max-abs amax gets the smallest e with amax <= 448 * 2^e,
 * clamped to [-127, 127] (e = 0 for an all-zero group); its codes are
 * E4M3(fl32(x * 2^-e)) rounded to nearest even with saturation.
 * Requirements: K % 128 == 0 (UNSUPPORTED); ldx, ldq >= K and ldsf >= R
 * (INVALID_ARG); x, q 16-byte aligned, ldx*sizeof(xt) and ldq multiples of 16,
 * sf 4-byte aligned (MISALIGNED; fp8bs_mx_gemm wants sf 16-byte aligned and
 * ldsf % 4 == 0).  R == 0 or K == 0 is a no-op.  One launch on the stream. */
fp8bs_status fp8bs_mx_quant_1x32(const void* x, fp8bs_dtype xt, int64_t R, int64_t K, int64_t ldx,
                                 uint8_t* q, int64_t ldq, uint32_t* sf, int64_t ldsf,
                                 void* stream);

/* MX GEMM: C[M x N] = sum over 32-deep K groups g of
 *   ( sum_{k in g} dec(A[m][k]) * dec(B[n][k]) ) * 2^(ea(m,g) + eb(n,g))
 * with the group exponents applied by the tensor cores (tcgen05 block-scaled
 * MMA), FP32 accumulation over all of K, BF16 (round to nearest even) or
 * FP32 output.  Same passages as fp8bs_mx_quant_1x32.
 *   A [M x K] codes (lda), B [N x K] codes (ldb), both K contiguous (device);
 *   sfa / sfb exponent words of A's and B's rows in the layout that
 *   fp8bs_mx_quant_1x32 writes (ldsfa >= M, ldsfb >= N);
 *   C [M x N] row-major, ldc elements (device, caller-owned).
 * Requirements: K % 128 == 0 and N % 16 == 0 (UNSUPPORTED); leading
 * dimensions as above (INVALID_ARG); A, B, C, sfa, sfb 16-byte aligned, lda
 * and ldb multiples of 16, ldc*sizeof(ct) a multiple of 16, ldsfa and ldsfb
 * multiples of 4 (MISALIGNED).  M == 0 or N == 0: no-op; K == 0: C = 0.
 * Asynchronous on the stream; allocates nothing; fp8bs_sync_status reports a
 * device-side timeout. */
fp8bs_status fp8bs_mx_gemm(int64_t M, int64_t N, int64_t K, const uint8_t* A, int64_t lda,
                           const uint32_t* sfa, int64_t ldsfa, const uint8_t* B, int64_t ldb,
                           const uint32_t* sfb, int64_t ldsfb, void* C, fp8bs_dtype ct,
                           int64_t ldc, void* stream);

/* Synchronize the stream, then report (and clear) the device error word of the
 * current device: FP8BS_ERR_DEVICE_TIMEOUT, FP8BS_ERR_DEVICE_BAD_ROUTING,
 * FP8BS_ERR_DEVICE_BAD_OFFSETS (in that order of precedence), FP8BS_ERR_CUDA
 * for a sticky CUDA error, else FP8BS_OK. */
fp8bs_status fp8bs_sync_status(void* stream);

/* Static string naming a status code. */
const char* fp8bs_status_string(fp8bs_status status);

/* Accumulation probe of the tensor cores (the page at why-be.why-be.co.kr,
 * accumulation-precision passage: on H800 the FP8 MMA keeps only about 14
 * bits of its accumulated sum).  Computes D[128][256] = A[128][K] * B[256][K]^T
 * over raw E4M3 codes (no scales) with K/32 tcgen05 kind::f8f6f4 MMAs
 * (M=128, N=256, K=32) accumulating in TMEM, and returns the FP32 result as
 * the hardware produced it, so the caller can compare it with the exact sum.
 *   a  [128][K] codes, row stride K bytes (device);  b [256][K] likewise;
 *   d  [128][256] fp32, row-major (device).
 * Requirements: K in {32, 64, 96, 128} (UNSUPPORTED); pointers non-NULL
 * (INVALID_ARG), d 4-byte aligned (MISALIGNED).  One CTA; asynchronous on
 * the stream; fp8bs_sync_status reports a device-side timeout. */
fp8bs_status fp8bs_probe_mma_f8f6f4(const uint8_t* a, const uint8_t* b, int64_t K, float* d,
                                    void* stream);

/* Test hook for the failure path: launch one CTA that waits on a barrier no
 * one arrives at, with a limit of limit_ns nanoseconds (1e3 .. 1e10).  The
 * wait gives up, records a timeout in the device error word and returns, so
 * fp8bs_sync_status() then reports FP8BS_ERR_DEVICE_TIMEOUT.  No trap, no
 * hang.  Not part of the method (the pages have no counterpart). */
fp8bs_status fp8bs_debug_timeout_probe(int64_t limit_ns, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* FP8BS_H */
