/*
 * q6mmq -- q6_K x int8 ("MMQ") prefill GEMM for GB300 (sm_103a), C ABI.
 *
 * The operation (pages of the minfer CUDA optimisation log on the q6_K GEMM):
 *   "r38 -- q6_K BT-style raw-byte mma kernel", Sec. 2.1 and 2.2: weights are
 *   q6_K super-blocks of 256 elements (ql[128] low nibbles, qh[64] high 2-bit
 *   fields, 16 int8 sub-block scales sc, one f16 scale d); the dequantised
 *   weight is d * sc[sub] * (q - 32); activations are int8 with one f32 scale
 *   da per 32 elements; the product is rescaled per 16-element sub-block with
 *   sum += da * (d * sc), and there is no dmin term.
 *
 *   Y[n][m] = sum_k (d*sc*(q-32))[m][k] * (da*xq)[n][k].
 *
 *   This library forms, per (n, m, 32-element chunk c), the exact integer
 *   S = sum over the chunk's two sub-blocks s of sc[s] * P[s], where
 *   P[s] = sum over the 16 elements of (q - 32) * xq, and then
 *   Y = sum over super-blocks of d * (sum over their chunks of da * S) in f32.
 *
 * Conventions for every call:
 *   - Pointers marked "device" are device memory owned by the caller; the
 *     library never frees or keeps them. Calls allocate nothing, except that
 *     the first call on a device allocates one 256-byte status block there,
 *     kept until process exit.
 *   - Every call is asynchronous on stream `s` (NULL = legacy default stream)
 *     and returns once the work is enqueued. Argument errors are detected on
 *     the host before anything is enqueued.
 *   - A device-side wait that exceeds its time limit (about one second) makes
 *     the kernel record a code and return early; q6_sync_status() reports it.
 *   - The current CUDA device must be compute capability 10.3 (GB300).
 *   - Return value: one of the Q6_* codes below; q6_last_error() gives a
 *     one-line text for the calling thread's last non-zero return.
 */
#ifndef Q6MMQ_H
#define Q6MMQ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *q6_stream_t; /* the same type as cudaStream_t */

#define Q6_OK 0
#define Q6_EINVAL 1   /* null pointer, bad size, K % 256 != 0, leading dimension too small */
#define Q6_EALIGN 2   /* a pointer or leading dimension breaks its stated alignment */
#define Q6_ESIZE 3    /* a size outside the supported range */
#define Q6_EARCH 4    /* the current device is not compute capability 10.3 */
#define Q6_ECUDA 5    /* a CUDA call failed */
#define Q6_ETIMEOUT 6 /* a bounded device-side wait expired (from q6_sync_status) */

/* Which kernels a q6k_mmq call ran (written to *path_out). */
#define Q6_PATH_NONE 0    /* nothing to do (N == 0) */
#define Q6_PATH_TC_RAW 1  /* unpack of the packed q6_K plane into the workspace + tensor-core GEMM */
#define Q6_PATH_TC_WEXP 2 /* conversion of the W_exp plane into the workspace + tensor-core GEMM */
#define Q6_PATH_SKINNY 3  /* few-token kernel for N <= Q6_SKINNY_MAX_N on the packed q6_K plane */
#define Q6_PATH_TC_WH 4   /* tensor-core GEMM on resident binary16 operand planes */
#define Q6_PATH_SYNC_WEXP 5 /* legacy mma.sync int8 GEMM on the W_exp plane (q6k_mmq_mma_sync) */
#define Q6_PATH_SKINNY_FUSED 6 /* quantiser and one/two-token GEMM in one kernel (q6k_mmq_f32) */
#define Q6_PATH_Q4K_TC_RAW 7 /* q4_K: unpack of the packed plane into the workspace + tensor-core GEMM */
#define Q6_PATH_Q4K_TC_WQ 8  /* q4_K: tensor-core GEMM on a resident binary16 operand plane */
#define Q6_PATH_TC_FUSED_RAW 9 /* q6k_mmq_f32_tc: unpack into the workspace + GEMM quantising X itself */
#define Q6_PATH_TC_FUSED_WH 10 /* q6k_mmq_f32_tc: GEMM quantising X itself, resident operand planes */
#define Q6_PATH_Q4K_SKINNY 11  /* q4_K: few-token kernels on the packed plane */
#define Q6_PATH_Q4K_SKINNY_FUSED 12 /* q4k_mmq_f32: quantiser and one/two-token GEMM in one kernel */

/* q4k_mmq runs N <= Q6_Q4K_SKINNY_MAX_N on the few-token kernels on the
 * packed plane: N <= Q6_Q4K_DP4A_MAX_N on dp4a (CUDA cores), more on the
 * warp-level f16 tensor path (measured on GB300, q4_K weights of 4096 x
 * 11008: dp4a 8.6 / 11.2 us at 1 / 2 tokens; the f16 kernel about 13-14 us
 * at 3-8 tokens and 17 us at 16, against about 53 us on the tensor cores from
 * the packed plane and 30 us from the resident operand plane). */
#define Q6_Q4K_SKINNY_MAX_N 16
#define Q6_Q4K_DP4A_MAX_N 2

/* q4k_mmq with Xq runs Q6_Q4K_SKINNY_MAX_N < N <= Q6_Q4K_GROUP_N on the
 * few-token f16 kernel whatever the weight source, and, without a resident
 * operand plane (wq NULL), N <= Q6_Q4K_GROUPS_MAX_N too, in token groups of
 * at most Q6_Q4K_GROUP_N (measured on GB300, 4096 x 11008: 21.6 / 24.4 / 39.2 /
 * 48.3 us at 17 / 32 / 48 / 64 tokens, against 52-55 us for the unpack and the tensor
 * cores, and 29-30 us for the tensor cores on the resident plane at 17-32
 * tokens). */
#define Q6_Q4K_GROUPS_MAX_N 64
#define Q6_Q4K_GROUP_N 32

/* q6k_mmq with Xq runs Q6_SKINNY_MAX_N < N <= Q6_SKINNY_GROUP_N on the
 * few-token kernels whatever the weight source, and, without resident operand
 * planes (wh NULL), N <= Q6_SKINNY_GROUPS_MAX_N too, in token groups of at
 * most Q6_SKINNY_GROUP_N (each group streams the 0.82-byte packed plane once;
 * measured on GB300, 4096 x 11008: 17 / 32 / 48 / 64 / 80 / 96 tokens in about
 * 23 / 27 / 44 / 53 / 70 / 78 us, against 77-80 us for unpacking 4 bytes a
 * weight and the tensor-core GEMM, and 37-38 us for the tensor cores on
 * resident planes at 17-32 tokens). */
#define Q6_SKINNY_GROUPS_MAX_N 96
#define Q6_SKINNY_GROUP_N 32

#define Q6_SKINNY_MAX_N 16
#define Q6_FUSED_MAX_N 2   /* tokens q6k_mmq_f32 takes */

/* Text of the calling thread's last error ("" if none). Owned by the library. */
const char *q6_last_error(void);

/* Q6_OK if the current device is compute capability 10.3, else Q6_EARCH. */
int q6_device_check(void);

/* Waits for stream `s`, then reads and clears this device's status word.
 * Returns Q6_OK, Q6_ETIMEOUT (a kernel gave up a bounded wait; the text names
 * the wait) or Q6_ECUDA (the stream itself reported an error). */
int q6_sync_status(q6_stream_t s);

/* Diagnostic: launches one single-warp kernel whose only work is a bounded
 * wait on a barrier that nothing completes, with a limit of `limit_ms`
 * milliseconds (1..2000). The kernel records the time-out in the status word
 * and returns, so a following q6_sync_status() reports Q6_ETIMEOUT and the
 * context stays usable. Used to test the time-out path without a fault. */
int q6_selftest_wait_timeout(int limit_ms, q6_stream_t s);

/* ------------------------------------------------------------------------
 * Activation quantisation (the activation prepass; "r38 -- q6_K BT-style
 * raw-byte mma kernel", Sec. 2.2 names its per-32 scale da).
 *
 * For token n and 32-element block c: amax = max|x|, da = amax/127 (f32),
 * xq = clamp(round_half_away(x / da), -127, 127) with an IEEE f32 division;
 * amax == 0 gives da = 0 and xq = 0. Inputs must be finite.
 *
 * Output layouts (all device, caller-allocated):
 *   Xq : int8 [N][K], row stride K.
 *   da : f32 [K/32][ldda], ldda = N rounded up to a multiple of 4;
 *        da[c * ldda + n]. Entries n >= N are left untouched.
 *   Xh : binary16 [N][K], row stride K; Xh[n][k] = (half)Xq[n][k] (exact).
 *        This is the operand plane the tensor-core GEMM reads. Optional.
 * -------------------------------------------------------------------- */

/* Sizes in bytes of the three outputs for an N x K activation, and ldda.
 * Any output pointer may be NULL. Q6_EINVAL if N < 0, K <= 0 or K % 256. */
int q8_act_plane_bytes(int N, int K, size_t *xq_bytes, size_t *da_bytes,
                       size_t *xh_bytes, int *ldda);

/* X: device f32 [N][ldx], ldx >= K, X and ldx*4 16-byte aligned.
 * da required; at least one of Xq and Xh (the other may be NULL: a prefill
 * caller that only runs the tensor-core GEMM needs Xh and da, the few-token
 * kernels need Xq and da). Xq, Xh, da 16-byte aligned. K % 256 == 0.
 * N == 0 is a no-op. */
int q8_quantize_act(const float *X, int N, int K, int ldx, int8_t *Xq, float *da,
                    uint16_t *Xh, q6_stream_t s);

/* Size in bytes of the block-sum pairs us of an N x K activation (below),
 * and their row length ldus = 32 * ceil(K / 512) f32 values. Either output
 * may be NULL. Q6_EINVAL if N < 0, K <= 0 or K % 256. */
int q8_act_sums_bytes(int N, int K, size_t *us_bytes, int *ldus);

/* The same as q8_quantize_act, and also the activation block sums the q4_K
 * GEMM needs ("r38 -- q6_K BT-style raw-byte mma kernel", Sec. 2.2: q4_K's
 * rescale has a second term with the activation block's sum), laid out as
 * the operand of the GEMM's min-term MMAs (kind::tf32):
 *   us : device f32 [N][ldus] (required, 16-byte aligned). For token n and
 *        block c (super-block b = c / 8, i = c % 8), the value
 *        v = da[c][n] * (sum of token n's 32 codes of block c), rounded to
 *        f32 once, is stored as the pair hi = v with its low 13 mantissa bits
 *        cleared, at us[n][16 b + i], and lo = v - hi (exact), at
 *        us[n][16 b + 8 + i]: hi + lo == v. An odd K/256 leaves the row's
 *        last 16 values zero. */
int q8_quantize_act_sums(const float *X, int N, int K, int ldx, int8_t *Xq, float *da,
                         uint16_t *Xh, float *us, q6_stream_t s);

/* ------------------------------------------------------------------------
 * Weight packing (load time; "r53 -- q6_K bundle: W_exp pre-expansion
 * plane", Sec. 2.3 and 3.2).
 *
 * raw: the bytes of an M x K q6_K weight in the GGUF layout: M rows, each
 *      K/256 consecutive 210-byte super-blocks (ql[128] @0, qh[64] @128,
 *      sc[16] int8 @192, d f16 little endian @208). No alignment needed.
 *      Device memory, or host memory the device reads directly: page-locked
 *      host memory (cudaHostAlloc / cudaHostRegister), or any host memory on
 *      a device that reads pageable memory (cudaDevAttrPageableMemoryAccess,
 *      e.g. Grace-Blackwell's coherent host memory); other pageable host
 *      memory gives Q6_EINVAL. The pack kernel reads raw asynchronously on
 *      stream s: host memory must stay valid until the stream has passed it.
 *
 * plane (device, 256-byte aligned, q6k_plane_bytes() bytes), four sub-planes
 * at 256-byte aligned offsets, in this order:
 *   qlh : uint8 [M][K/128][96]. For each 128-element half h of a row
 *         (super-block h/2, half h%2): bytes 0..63 = ql[64*(h%2) .. +63],
 *         bytes 64..95 = qh[32*(h%2) .. +31] of that super-block.
 *         Row stride 3*K/4 bytes.
 *   sc  : int8 [M][K/16], the raw sub-block scales.
 *   d   : binary16 bits [M][ldd], the raw super-block scales; row stride
 *         ldd = K/256 rounded up to a multiple of 8 (16 bytes), padding zero.
 *   dT  : f32 [K/256][ldm], ldm = M rounded up to a multiple of 4: the
 *         super-block scales as f32 (exact), transposed; rows M..ldm-1 zero.
 * wexp (device, optional, 16-byte aligned): int8 [M][K], row stride K, the
 *      centered values v = q - 32 in [-32, 31] (the W_exp plane).
 * wh   (device, optional, 16-byte aligned): binary16 [2][M][K], the two
 *      operand planes the tensor-core GEMM reads (4 bytes per weight), with
 *      the sub-block scale folded in and split so both stay exact:
 *      wh[0][m][k] = 16 * floor(sc/16) * v and wh[1][m][k] = (sc mod 16) * v,
 *      sc the scale of k's sub-block; wh[0] + wh[1] = sc * v. (Zero may be
 *      stored as -0.)
 * -------------------------------------------------------------------- */

/* Byte sizes of the packed plane and of the W_exp plane (the wh planes are
 * four times the W_exp size). Either pointer may be NULL. */
int q6k_plane_bytes(int M, int K, size_t *plane_bytes, size_t *wexp_bytes);

/* Fills `plane` (and `wexp`, `wh` when not NULL) from `raw`. M > 0,
 * K % 256 == 0. */
int q6k_pack_weights(const uint8_t *raw, int M, int K, void *plane, int8_t *wexp,
                     uint16_t *wh, q6_stream_t s);

/* The weight unpack pass alone: writes the binary16 operand planes wh
 * [2][M][K] (the layout described above) from wexp and the plane's sc
 * sub-plane when wexp is not NULL, else from the packed plane's qlh and sc
 * sub-planes ("r41 -- q6_K B-expand widened to uint4 group loads", Sec. 3.2:
 * 16-element groups from one 16-byte ql run and one 16-byte qh run). plane is
 * required in both cases. q6k_mmq runs this into its workspace when it gets
 * no wh planes. */
int q6k_unpack_weights(const void *plane, const int8_t *wexp, int M, int K, uint16_t *wh,
                       q6_stream_t s);

/* ------------------------------------------------------------------------
 * The GEMM.  Y[n][m] for n < N, m < M (f32, row stride ldy >= M, device).
 *
 *   plane : packed weights from q6k_pack_weights (required).
 *   wexp, wh : the optional planes from q6k_pack_weights, or NULL.
 *   Xq, da: quantised activations (layouts above). Xq is read by the
 *           few-token kernels (N <= Q6_SKINNY_MAX_N: dp4a on the CUDA cores
 *           for one or two tokens, exact f16 mma.sync for 3..16 tokens; both
 *           stream the packed plane once), and, on token groups of at most
 *           Q6_SKINNY_GROUP_N (the same mma.sync kernel holds 17..32 tokens),
 *           for up to Q6_SKINNY_GROUP_N tokens whatever the weight source and
 *           without wh for up to Q6_SKINNY_GROUPS_MAX_N tokens.
 *   Xh    : the binary16 operand plane; required when N > Q6_SKINNY_MAX_N,
 *           unless the token groups apply.
 *   workspace : device scratch, 256-byte aligned, of at least
 *           q6k_mmq_workspace_bytes() bytes when N > Q6_SKINNY_MAX_N and either
 *           wh is NULL or partials is not NULL: the weights are first unpacked
 *           there (from wexp when given, else from the packed plane) into the
 *           two binary16 operand planes (4 * M * K bytes), and the debug
 *           passes below reuse it. After those bytes (rounded up to 256) it
 *           may also hold the K-part partial sums of a call with few tiles
 *           (q6k_tc_part_bytes(); with resident wh planes that is all the
 *           workspace is used for): without room for them the call runs
 *           unsplit, with the same Y up to rounding and slower. Its contents
 *           after the call are unspecified.
 *   partials : NULL, or device int32 [N][M][K/16] that receives every exact
 *           sub-block partial P[n][m][s] = sum over the 16 elements k of
 *           sub-block s of (q[m][k] - 32) * xq[n][k] (the debug mode of "r38
 *           -- q6_K BT-style raw-byte mma kernel", Sec. 2.4: one int32 per
 *           sub-block; slower). The few-token kernels and the mma.sync path
 *           write the P they form; the tensor-core path, whose operands carry
 *           the sub-block scale, forms them in two more GEMM launches on
 *           planes unpacked with unit scale (W_hi = 0, W_lo = v on the
 *           sub-blocks of one parity, 0 on the others) in the workspace.
 *   chunk_sums : NULL, or device int32 [N][M][K/32] that receives the exact
 *           integer the kernel itself forms per 32-element chunk c,
 *           S[n][m][c] = sc[2c] * P[2c] + sc[2c+1] * P[2c+1] (debug).
 *   path_out : NULL or receives a Q6_PATH_* code.
 * Alignment: plane, workspace 256 B; Xh, da, wexp, wh, Xq 16 B; Y, partials,
 * chunk_sums 4 B. Q6_ESIZE when a needed workspace is missing or too small.
 *
 * Work split: the tensor-core path walks 128 x 128 output tiles with one
 * persistent CTA per SM. When the last round of tiles would leave more than
 * half of the SMs idle, each of its tiles is computed as two halves of its
 * super-blocks on two SMs; a small kernel first zeroes those tiles of Y and
 * both halves add into it. Two addends onto zero give the same sum in either
 * order, so Y stays deterministic; it can differ from the unsplit sum by
 * rounding only (the partials are unaffected).
 * -------------------------------------------------------------------- */
int q6k_mmq_workspace_bytes(int M, int K, int N, size_t *bytes);

/* The number of kernels one q6k_mmq call launches for this shape on the
 * calling thread's current device: 0 for N == 0; 1 on the skinny path
 * (N <= Q6_SKINNY_MAX_N); ceil(N / Q6_SKINNY_GROUP_N) on token groups
 * (N <= Q6_SKINNY_GROUP_N, or has_wh == 0 and N <= Q6_SKINNY_GROUPS_MAX_N,
 * counted as if Xq is given);
 * otherwise 1 for the tensor-core GEMM, plus 1 when
 * either work split above applies (the zeroing of the split last round, or
 * the addition of the K parts, counted as if the workspace had room for
 * them), plus 1 when the weights are unpacked into the workspace first
 * (has_wh == 0). Q6_EINVAL on bad sizes or a NULL launches; Q6_EARCH /
 * Q6_ECUDA as for the other calls. */
int q6k_mmq_launches(int M, int K, int N, int has_wh, int *launches);

int q6k_mmq(const void *plane, const int8_t *wexp, const uint16_t *wh, int M, int K,
            const int8_t *Xq, const float *da, const uint16_t *Xh, int N, float *Y, int ldy,
            void *workspace, size_t workspace_bytes, int32_t *partials, int32_t *chunk_sums,
            int *path_out, q6_stream_t s);

/* ------------------------------------------------------------------------
 * The pages' own route on the legacy warp-level tensor path, kept as a
 * measured comparison point for q6k_mmq ("r38 -- q6_K BT-style raw-byte mma
 * kernel", Sec. 2.2-2.4; "r53 -- q6_K bundle: W_exp pre-expansion plane",
 * Sec. 2.3): exact int32 sub-block partials from int8 mma.sync on the W_exp
 * plane and Xq, sc folded per 32-element chunk in integers, f32 rescale.
 * Same result contract as q6k_mmq (Y within the same tolerance; partials and
 * chunk_sums, when not NULL, are the same int32 [N][M][K/16] sub-block
 * partials and [N][M][K/32] chunk sums, written by the GEMM kernel itself).
 *
 *   plane : packed weights (its sc and dT sub-planes are read); required.
 *   wexp  : the W_exp plane; required.
 *   Xq, da: quantised activations (any N >= 0).
 * Alignment: plane 256 B; wexp, Xq, da 16 B; Y, partials, chunk_sums 4 B.
 * Allocates nothing. path_out receives Q6_PATH_SYNC_WEXP (or Q6_PATH_NONE for
 * N == 0).
 * -------------------------------------------------------------------- */
int q6k_mmq_mma_sync(const void *plane, const int8_t *wexp, int M, int K, const int8_t *Xq,
                     const float *da, int N, float *Y, int ldy, int32_t *partials,
                     int32_t *chunk_sums, int *path_out, q6_stream_t s);

/* ------------------------------------------------------------------------
 * For callers that cannot allocate device memory when they make this call
 * (code under a fixed budget or pool that forbids new allocations, or a
 * latency-critical path that must never enter the allocator). The pages have
 * no counterpart: this is an alternative way to run q6k_mmq.
 *
 * Computes what q6k_mmq computes with the weights unpacked per call (from
 * wexp when not NULL, else from the packed plane; no resident wh plane and no
 * workspace argument), but its scratch is one static device array of the
 * library: 256 bytes for the kernel's status word plus 64 MiB for the
 * two unpacked binary16 operand planes, so when it unpacks (N >
 * Q6_SKINNY_MAX_N, and not the token groups that q6k_mmq also runs for N <=
 * Q6_SKINNY_GROUPS_MAX_N given Xq) it needs M * K <= 16,777,216 (a 4096 x
 * 4096 layer) and returns Q6_ESIZE otherwise. Nothing on this path
 * allocates; no debug outputs.
 *
 * The array is held by every GPU that loads this part of the library until
 * the process exits. All calls share it and it keeps the last call's
 * contents: calls that overlap on the GPU race on it. The status word is
 * cleared on the call's stream at the start of every call; a bounded-wait
 * time-out is recorded there and q6k_mmq_noalloc_status() reports it. The
 * first call on a device does the set-up (architecture check, kernel
 * attributes, the array's device address) and should come before any stream
 * capture. */
int q6k_mmq_noalloc(const void *plane, const int8_t *wexp, int M, int K, const int8_t *Xq,
                    const float *da, const uint16_t *Xh, int N, float *Y, int ldy, int *path_out,
                    q6_stream_t s);

/* The status of the q6k_mmq_noalloc calls on this device: waits for stream
 * `s`, then reads and clears the status word in the static array. Returns
 * Q6_OK, Q6_ETIMEOUT (a kernel gave up a bounded wait; the text names the
 * wait) or Q6_ECUDA. Allocates nothing. No counterpart in the pages. */
int q6k_mmq_noalloc_status(q6_stream_t s);

/* ------------------------------------------------------------------------
 * One or two tokens straight from f32 activations, in one kernel launch:
 * Y = what q8_quantize_act followed by q6k_mmq gives for the same X (the
 * per-32 quantisation of "r38 -- q6_K BT-style raw-byte mma kernel" Sec. 2.2
 * with the same arithmetic, then the q6_K GEMM of Sec. 2.1-2.2), without
 * writing the codes and scales to memory. For decode steps, where the
 * quantiser's separate launch is a large share of the step.
 *
 *   plane : packed weights from q6k_pack_weights (device, 256-byte aligned).
 *   X     : device f32 [N][ldx], ldx >= K; X 16-byte aligned, ldx % 4 == 0.
 *   N     : 0 .. Q6_FUSED_MAX_N (more tokens: q8_quantize_act + q6k_mmq).
 *   Y     : device f32 [N][ldy], ldy >= M, 4-byte aligned.
 *   K     : K % 256 == 0 and N * K * 9 / 8 <= 232,448 (the codes and scales
 *           of X staged in shared memory): K <= 103,168 for two tokens,
 *           206,592 for one; Q6_ESIZE beyond.
 *   path_out : NULL or receives Q6_PATH_SKINNY_FUSED (Q6_PATH_NONE for N == 0).
 * Errors: Q6_EINVAL, Q6_EALIGN, Q6_ESIZE, Q6_EARCH, Q6_ECUDA as above; no
 * allocation, no bounded waits, asynchronous on s. */
int q6k_mmq_f32(const void *plane, int M, int K, const float *X, int ldx, int N, float *Y,
                int ldy, int *path_out, q6_stream_t s);

/* The tensor-core GEMM from f32 activations, with the quantiser fused into
 * the GEMM's producer: the kernel reads X, forms each 32-element block's da
 * and binary16 codes in shared memory (bit for bit those of
 * q8_quantize_act), and runs the GEMM on them; no Xh or da plane is written.
 * This is the inverse of the pages' prepass ("r38 -- q6_K BT-style raw-byte
 * mma kernel", Sec. 1: r34 moved the A-side transform out of the GEMM into a
 * prepass). Y is bit for bit that of q8_quantize_act + q6k_mmq on the
 * tensor-core path (N > Q6_SKINNY_MAX_N), and for any N >= 1 within the
 * tolerance of the oracle. The kernel quantises every activation block once
 * per 128-row weight band (M / 128 times), against once for the separate
 * quantiser.
 *   plane : packed q6_K plane (required, for d); wh : resident operand planes
 *           [2][M][K] or NULL (then they are unpacked into the workspace).
 *   X : device f32 [N][ldx], 16-byte aligned, ldx >= K, ldx % 4 == 0.
 *   workspace : 256-byte aligned, at least 4 * M * K bytes when wh is NULL.
 *   path_out : NULL or receives Q6_PATH_TC_FUSED_RAW / Q6_PATH_TC_FUSED_WH.
 * Errors as for q6k_mmq. */
int q6k_mmq_f32_tc(const void *plane, const uint16_t *wh, int M, int K, const float *X, int ldx,
                   int N, float *Y, int ldy, void *workspace, size_t workspace_bytes,
                   int *path_out, q6_stream_t s);

/* ------------------------------------------------------------------------
 * The q4_K x int8 GEMM ("r18: Load-time B pre-expansion -- staging becomes a
 * bulk copy", Sec. 1 and 3.2: the 144-byte block and its per-chunk pair
 * (d * sc, -dmin * m); "r38 -- q6_K BT-style raw-byte mma kernel", Sec. 2.2:
 * the two-term rescale). Weights are q4_K super-blocks of 256 elements in 8
 * sub-blocks of 32; the dequantised weight is d * sc[j] * q - dmin * m[j]
 * (q the raw nibble 0..15, sc and m 6-bit):
 *
 *   Y[n][m] = sum over sub-blocks c of da[c][n] * (d * sc[c] * P[n][m][c]
 *                                                  - dmin * m[c] * S[n][c]),
 *   P = sum over the 32 elements of q * xq,  S = sum of the 32 xq.
 *
 * raw (q4k_pack_weights): M rows of K/256 consecutive 144-byte blocks in the
 *      GGUF layout: d (f16) @0, dmin (f16) @2, 12 bytes of packed 6-bit
 *      scales and mins @4, 128 nibble bytes @16 (nibble pair p: the 32 bytes
 *      at 16 + 32 p, sub-block 2p in the low nibbles and 2p + 1 in the high
 *      ones). The 12-byte packing, which the pages call but do not print, is
 *      read as GGUF's: sub-blocks j < 4 take the low 6 bits of bytes j
 *      (scale) and j + 4 (min); sub-blocks j >= 4 take the nibbles of byte
 *      j + 4 (low: scale, high: min) as their low 4 bits and the top 2 bits
 *      of bytes j - 4 (scale) and j (min) as bits 4-5. Device memory or host
 *      memory the device reads, as for q6k_pack_weights.
 * plane (device, 256-byte aligned, q4k_plane_bytes() bytes), sub-planes at
 *      256-byte aligned offsets: qs uint8 [M][K/2] (the nibble bytes as they
 *      are), sc uint8 [M][K/32], m uint8 [M][K/32] (decoded), dT f32
 *      [K/256][ldm] (d, transposed, ldm = M rounded up to 4), mv f32
 *      [M][ldus] (dmin * m of every sub-block, at most 17 significant bits,
 *      as the exact pair hi + lo in the layout of the activations' us, see
 *      q8_quantize_act_sums; ldus = 32 * ceil(K / 512)), ddm f32 [M][K/256][2]
 *      ((d, dmin) of every super-block, for the few-token kernel); padding
 *      is zero.
 * wq (device, optional, 16-byte aligned): the binary16 operand plane [M][K]
 *      the tensor-core GEMM reads, sc * q (at most 945: exact).
 * -------------------------------------------------------------------- */

/* Bytes of the packed q4_K plane and of the wq plane (2 * M * K). */
int q4k_plane_bytes(int M, int K, size_t *plane_bytes, size_t *wq_bytes);

/* Fills plane (and wq when not NULL) from raw. M > 0, K % 256 == 0. */
int q4k_pack_weights(const uint8_t *raw, int M, int K, void *plane, uint16_t *wq,
                     q6_stream_t s);

/* The unpack pass alone: wq [M][K] from the packed plane. */
int q4k_unpack_weights(const void *plane, int M, int K, uint16_t *wq, q6_stream_t s);

/* One or two tokens of the q4_K GEMM straight from f32 activations, in one
 * kernel launch: Y = what q8_quantize_act_sums followed by q4k_mmq gives for
 * the same X (bit for bit), without writing the codes, scales and block sums
 * to memory; the q4_K counterpart of q6k_mmq_f32.
 *   plane : the packed q4_K plane (device, 256-byte aligned).
 *   X     : device f32 [N][ldx], ldx >= K; X 16-byte aligned, ldx % 4 == 0.
 *   N     : 0 .. Q6_FUSED_MAX_N (more tokens: q8_quantize_act_sums + q4k_mmq).
 *   Y     : device f32 [N][ldy], ldy >= M, 4-byte aligned.
 *   K     : K % 256 == 0 and N * K * 5 / 4 <= 232,448 (the codes, scales and
 *           block sums of X staged in shared memory): K <= 92,928 for two
 *           tokens, 185,856 for one; Q6_ESIZE beyond.
 *   path_out : NULL or receives Q6_PATH_Q4K_SKINNY_FUSED (Q6_PATH_NONE for
 *           N == 0).
 * Errors: Q6_EINVAL, Q6_EALIGN, Q6_ESIZE, Q6_EARCH, Q6_ECUDA as above; no
 * allocation, no bounded waits, asynchronous on s. */
int q4k_mmq_f32(const void *plane, int M, int K, const float *X, int ldx, int N, float *Y,
                int ldy, int *path_out, q6_stream_t s);

/* The q4_K GEMM. N > Q6_Q4K_SKINNY_MAX_N runs on the tensor cores; fewer
 * tokens run weight-streaming few-token kernels on the packed plane (about
 * 0.59 byte per weight; wq and the workspace are not used): dp4a for N <=
 * Q6_Q4K_DP4A_MAX_N, exact f16 mma.sync beyond. With Xq, up to
 * Q6_Q4K_GROUP_N tokens (and, without wq, up to Q6_Q4K_GROUPS_MAX_N) run the
 * f16 few-token kernel on token groups of at most Q6_Q4K_GROUP_N instead of
 * the tensor cores.
 *   plane : the packed q4_K plane (required); wq : resident operand plane or
 *           NULL (then it is unpacked into the workspace first).
 *   Xq, Xh, da, us : from q8_quantize_act_sums (int8 codes, binary16 codes,
 *           scales, block-sum pairs); Xq is required for N <=
 *           Q6_Q4K_SKINNY_MAX_N and Xh for more tokens (unless the token
 *           groups run). The min term sum_c us * (dmin * m) runs as tf32
 *           products of the hi/lo pairs on the tensor cores and in the f16
 *           few-token kernel (each product exact in f32; us's pair is within
 *           2^-21 |us| of it); the dp4a kernel adds each pair back to us (exact).
 *   workspace : device, 256-byte aligned, at least 2 * M * K bytes on the
 *           tensor-core path when wq is NULL or partials is not NULL; contents
 *           afterwards unspecified.
 *   partials : NULL, or device int32 [N][M][K/32] that receives every exact
 *           P = sum over a sub-block of q * xq (debug: on the tensor cores one
 *           more GEMM launch on the plane of the raw nibbles, unpacked in the
 *           workspace; the few-token kernels write them from their dot
 *           products).
 *   path_out : NULL or receives Q6_PATH_Q4K_TC_RAW / Q6_PATH_Q4K_TC_WQ /
 *           Q6_PATH_Q4K_SKINNY.
 * Alignment: plane, workspace 256 B; Xq, Xh, da, us, wq 16 B; Y, partials 4 B.
 * Errors as for q6k_mmq. */
int q4k_mmq(const void *plane, const uint16_t *wq, int M, int K, const int8_t *Xq,
            const uint16_t *Xh, const float *da, const float *us, int N, float *Y, int ldy,
            void *workspace, size_t workspace_bytes, int32_t *partials, int *path_out,
            q6_stream_t s);

#ifdef __cplusplus
}
#endif

#endif /* Q6MMQ_H */
