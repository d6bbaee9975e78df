/*
 * qmv.h - C ABI of libqmv: fused dequantize-and-matvec for the decode step of
 * a compressed LLM, on one GB300 (sm_103a).
 *
 * The operation every entry point serves is y = W_hat x at batch 1 up to a
 * small number M of speculative-verification tokens, where W_hat is a packed,
 * quantized N x K weight matrix and x holds M bf16 activation rows. Decoding at
 * low batch reads every active weight once per token, so the packed weight
 * stream is the cost ("Nemotron 3.5 Bolt", why-only-weights section; "Cassandra",
 * section 2: FFN weight loading dominates decode).
 *
 * Conventions shared by every call:
 *  - Device pointers point into memory the caller allocated (for example with
 *    torch); the library never allocates or frees device memory. Host pointers
 *    are marked "host".
 *  - Every device buffer must be 16-byte aligned; activation row strides must
 *    keep each row 16-byte aligned (ldx a multiple of 8 bf16 elements).
 *  - Calls are asynchronous on the caller's CUDA stream (`stream` is a
 *    cudaStream_t passed as void*; NULL = legacy default stream) and never
 *    synchronize. They return a qmv_status and never throw or abort.
 *  - Argument errors are found on the host before any launch and leave every
 *    output untouched. Corrupt packed data found by a kernel sets a per-device
 *    error word (read with qmv_check_status); the kernel still ends normally.
 *  - qmv_last_error() gives a message for the calling thread's last failure.
 *  - W is N x K (output rows x input columns). Quantization blocks/groups are
 *    128 consecutive columns of one row. x is bf16 [M][ldx], y is fp32 [M][ldy].
 */
#ifndef QMV_H
#define QMV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define QMV_ABI_VERSION 1
#define QMV_GROUP 128          /* block/group size along K for ternary and INT4 */
#define QMV_MAX_SECTIONS 8
#define QMV_MAX_M 16           /* activation rows per call */
#define QMV_MAX_BATCH 448      /* matvecs per qmv_run_batch call */

typedef enum {
  QMV_OK = 0,
  QMV_ERR_ARG = -1,          /* bad argument, size or descriptor */
  QMV_ERR_ALIGN = -2,        /* pointer or stride misaligned */
  QMV_ERR_UNSUPPORTED = -3,  /* valid request this build does not serve */
  QMV_ERR_CORRUPT = -4,      /* a kernel met packed data that breaks the format */
  QMV_ERR_CUDA = -5,         /* a CUDA runtime call failed (message has the CUDA error) */
  QMV_ERR_TIMEOUT = -6       /* a kernel's bounded device-side wait (a copy completion) gave up
                                after its time limit; recorded in the device error word, read
                                with qmv_check_status; the kernel's outputs are then invalid */
} qmv_status;

typedef enum {
  QMV_TERNARY2 = 1,          /* block-128 absmean ternary, 2 bits + fp16 scale per block */
  QMV_INT4 = 2,              /* group-128 absmax/7 INT4, 4 bits + fp16 scale per group */
  QMV_CASS = 3,              /* Cassandra lossless bf16 split (speculation + verification) */
  QMV_CASS_MX = 4,           /* Cassandra-2: the split with MX shared exponents (slightly lossy) */
  QMV_TERNARY2_SPARSE = 5,   /* ternary with flagged all-zero tiles left out */
  QMV_TERNARY2_LUT = 6,      /* QMV_TERNARY2's codes and scales in the byte-lookup layout (M = 1) */
  QMV_INT4_LUT = 7           /* QMV_INT4's codes and scales in the byte-lookup layout (M = 1) */
} qmv_format;

/*
 * Layout descriptor of one packed matrix: a contiguous buffer of sections,
 * each starting on a 256-byte boundary (off[i] bytes from the start).
 *
 * QMV_TERNARY2 ("Ternary Bonsai 2", section 1.2, block_ternary) and
 * QMV_INT4 ("GPT-5.4 ..." section 3.2, group-wise quantization):
 *   0 codes : row-group records. Rows go in groups of 16 (the last group
 *             padded with zero codes), columns in steps of 1024 (8 blocks of
 *             128, the last step possibly fewer: nbk = min(8, K/128 - 8s)).
 *             Record (group g, step s) = the 16 rows' code blocks of that
 *             step, row after row; group g starts at byte g*16*K*bits/8 and
 *             step s inside it at s*16*8*block_bytes. A block is 8 (ternary)
 *             or 16 (INT4) uint32 words. Ternary word of columns k0..k0+15:
 *             column r = k%16 at bit r (r even) or 15+r (r odd); code 00 = 0,
 *             01 = +1, 10 = -1 (11 is invalid). INT4 word of columns
 *             k0..k0+7: column r = k%8 at bit 2r (r even) or 14+2r (r odd);
 *             4-bit two's complement, -7..7.
 *   1 scales: fp16 scales (ternary fp16(mean|w| + 1e-8), INT4 fp16(max|w| / 7)
 *             of each block/group) in the record order of the codes: record
 *             (group g, step s) is 16 rows x 8 scales, 256 bytes, so the scale
 *             of (row n, block b) is element ((n/16)*S + b/8)*128 + (n%16)*8 + b%8
 *             with S = ceil(K/1024); rows past N and blocks past K/128 hold 0.
 * QMV_CASS ("Cassandra", sections 3.1-3.3):
 *   0 bitmap : N x K/32 uint32, bit j%32 of word j/32 set = value (n, j) kept
 *   1 signmant: N x K/16 uint32, nibble i = S<<3 | (M>>4) of the i-th kept value
 *   2 expstream: unary exponent codes (rank r = r zeros then a one), bits
 *             LSB-first in uint32 words, each row starting 16-byte aligned
 *   3 rowstart: N+1 uint32, first stream word of each row (last = total)
 *   4 codebook: 256 bytes, codebook[rank] = exponent field E
 *   5 pruned : N x K/2 uint16, raw bf16 bits of the pruned values
 *   6 mlo    : N x K/16 uint32, nibble i = M & 0xF of the i-th kept value
 *   Sections 0-4 are the speculation data, 5-6 the verification data.
 * QMV_CASS_MX ("Cassandra", section 3.3, the MX route of Cassandra-2): the
 * same Wanda bitmap and raw pruned values; the kept values of a row, in column
 * order, form groups of 32 that share their largest exponent g (e = max(E, 1)
 * per value); each value's 8-bit significand (128 + M, or M when E = 0) is
 * shifted right by g - e (truncated), giving A. Draft value (-1)^S * (A >> 4)
 * * 2^(g - 130), target value (-1)^S * A * 2^(g - 134): exact where e = g,
 * below the original by less than 2^(g - 134) elsewhere. K % 64 == 0.
 *   0 bitmap : N x K/32 uint32 (as QMV_CASS)
 *   1 gexp   : N x K/64 uint8, shared exponent of each group
 *   2 signs  : N x K/64 uint32, bit i%32 of word i/32 = S of kept value i
 *   3 dnib   : N x K/16 uint32, nibble i = A >> 4 of kept value i
 *   4 lnib   : N x K/16 uint32, nibble i = A & 15 of kept value i
 *   5 pruned : N x K/2 uint16, raw bf16 bits of the pruned values
 *   Sections 0-3 are the speculation data (3.625 bits per weight), 4-5 the
 *   verification data. group = 32.
 * QMV_TERNARY2_SPARSE ("Ternary Bonsai 2", 1.1, 3.3-3.4, 5.5: all-zero blocks
 * flagged with scale 1, structured block sparsity with a sparse index): the
 * codes of QMV_TERNARY2, in which every tile of 16 rows (one row group) x 128
 * columns whose codes are all zero is flagged and left out. n_symbols holds T,
 * the number of stored tiles; G = ceil(N/16), KB = K/128.
 *   0 tilemap  : G x ceil(KB/32) uint32, bit b%32 of word b/32 = tile (g, b) stored
 *   1 tilestart: G+1 uint32, stored tiles before group g (last = T)
 *   2 tileblock: T uint16, block index of each stored tile, group by group
 *   3 codes    : per group, records of up to 8 stored tiles in column order; a
 *                record is the 16 rows' code blocks of its tiles, row after row
 *   4 scales   : T x 16 fp16, the 16 rows' scales of each stored tile (1.0 for
 *                an all-zero block of a real row, 0 for padding rows)
 * QMV_TERNARY2_LUT ("Ternary Bonsai 2", section 1.2, block_ternary: the same
 * codes and fp16 scales as QMV_TERNARY2, arranged for the byte-lookup matvec
 * at one activation row). Rows go in NG = ceil(N/32) groups of 32 (the last
 * padded with zero codes and zero scales); KB = K/128 blocks.
 *   0 codes : NG * KB * 1024 bytes. A code byte holds the codes of four
 *             consecutive columns 4c..4c+3 of a block, column 4c + i at bits
 *             2i..2i+1 (00 = 0, 01 = +1, 10 = -1; 11 is invalid). The 32 bytes
 *             of (row n, block b) are rotated by n % 32: byte t holds column
 *             group c = (t + n) % 32. They lie in the 1024-byte record of
 *             (block b, row group n / 32), which starts at (b * NG + n / 32) *
 *             1024; inside it byte t of row n is at (t / 16) * 512 + (n % 32)
 *             * 16 + t % 16.
 *   1 scales: fp16 [KB][NG * 32]; the scale of (row n, block b) is element
 *             b * NG * 32 + n.
 * QMV_INT4_LUT ("GPT-5.4 ..." section 3.2: the same codes and fp16 scales as
 * QMV_INT4, arranged for the byte-lookup matvec at one activation row). Rows go
 * in NG = ceil(N/32) groups of 32 (the last padded with zero codes and zero
 * scales); KB = K/128 blocks.
 *   0 codes : NG * KB * 2048 bytes. Code byte p of a row's block holds columns
 *             2p (low nibble) and 2p + 1 (high nibble), 4-bit two's complement.
 *             A row's 64 bytes of a block are two halves of 32, each rotated by
 *             n % 32: position t < 32 holds byte (t + n) % 32, position t >= 32
 *             byte 32 + (t - 32 + n) % 32. They lie in the 2048-byte record of
 *             (block b, row group n / 32), which starts at (b * NG + n / 32) *
 *             2048; inside it position t of row n is at (t / 16) * 512 + (n % 32)
 *             * 16 + t % 16.
 *   1 scales: fp16 [KB][NG * 32], as QMV_TERNARY2_LUT.
 */
typedef struct {
  uint32_t abi_version;      /* QMV_ABI_VERSION */
  uint32_t format;           /* qmv_format */
  int64_t N, K;
  int32_t group;             /* 128 for ternary/INT4, 0 for Cassandra, 32 for Cassandra-2 (MX) */
  int32_t n_symbols;         /* Cassandra: number of codebook entries in use */
  int64_t off[QMV_MAX_SECTIONS];
  int64_t bytes[QMV_MAX_SECTIONS];
  int64_t total_bytes;       /* size of the whole packed buffer */
  uint64_t flags;            /* 0, or one QMV_FLAG_PATH_* bit (ternary/INT4 matvec) */
} qmv_desc;

/*
 * Kernel choice of the ternary/INT4 matvec entry points (qmv_desc.flags; the
 * packers leave it 0). With 0 the library picks: the tensor-core kernel
 * (mma.sync m16n8k16 on bf16, decode cost independent of M) for INT4 and for
 * ternary from M = 2, the fp16-FMA kernel (cost grows with M) for ternary at
 * M = 1. Setting one bit forces a kernel, for testing and tuning; both path bits
 * set is QMV_ERR_ARG. Results of both kernels satisfy the same error bound and
 * are reproducible bit for bit.
 */
#define QMV_FLAG_PATH_FMA 1u
#define QMV_FLAG_PATH_MMA 2u
/*
 * Testing only (ternary/INT4 matvec): the kernel's first wait is on a barrier
 * that nothing completes, limited to 1 ms, before any copy is issued. The wait
 * gives up, the kernel records QMV_ERR_TIMEOUT in the device error word and
 * ends without writing y, and qmv_check_status returns QMV_ERR_TIMEOUT. It
 * shows how a lost copy is reported without making the GPU fault. Any other
 * unknown flag bit is QMV_ERR_ARG.
 */
#define QMV_FLAG_TEST_WAIT_TIMEOUT 0x100u

/* One matvec of a batch: y[M][ldy] = W x[M][ldx] for the matrix packed in w. */
typedef struct {
  const qmv_desc* desc;      /* host pointer */
  const void* w;             /* device: packed buffer */
  const void* x;             /* device: bf16 [M][ldx] */
  float* y;                  /* device: fp32 [M][ldy] */
  int64_t ldx, ldy;
} qmv_task;

/*
 * Layout math only (host, no GPU needed): fill `out` for a ternary or INT4
 * matrix (either layout) of N x K with the given group (must be 128). K must be a positive
 * multiple of 128 and N positive; for QMV_CASS_MX (group 32) K must be a
 * multiple of 64. Returns QMV_ERR_UNSUPPORTED for QMV_CASS, whose stream
 * length depends on the data (use cass_pack_host).
 */
int qmv_pack_desc(int format, int64_t N, int64_t K, int32_t group, qmv_desc* out);

/*
 * Quantize and pack on the GPU (offline step). w: device fp32 [N][K] row-major.
 * qmv_pack_ternary writes QMV_TERNARY2 or QMV_TERNARY2_LUT, qmv_pack_int4
 * QMV_INT4 or QMV_INT4_LUT, after desc->format.
 * packed: device buffer of desc->total_bytes. Ternary follows block_ternary
 * ("Ternary Bonsai 2", 1.2): scale* = (sum_k |w_k|)/128 + 1e-8 summed in float64
 * in column order, q = clamp(rint(w/scale*), -1, 1) in float64, stored scale =
 * fp16(scale*) rounded to nearest even. INT4 ("GPT-5.4", 3.2): scale* =
 * max|w|/7 in float64, q = clamp(rint(w/scale*), -7, 7); an all-zero group
 * stores q = 0 and scale 0. Output bytes are fully determined by w.
 */
int qmv_pack_ternary(const qmv_desc* desc, const float* w, void* packed, void* stream);
int qmv_pack_int4(const qmv_desc* desc, const float* w, void* packed, void* stream);

/*
 * Flagged sparse ternary packer (host): dense_packed is a host copy of a
 * QMV_TERNARY2 buffer described by `dense`; desc receives the
 * QMV_TERNARY2_SPARSE layout (out == NULL: size query only) and out (host,
 * out_capacity >= desc->total_bytes) the buffer: tiles whose 16 x 128 codes are
 * all zero are left out, an all-zero block of a stored tile gets the scale 1.0.
 */
int qmv_sparse_pack_host(const qmv_desc* dense, const void* dense_packed, qmv_desc* desc, void* out,
                         int64_t out_capacity);

/*
 * Decode a packed ternary (QMV_TERNARY2 or QMV_TERNARY2_LUT) or INT4 (QMV_INT4 or QMV_INT4_LUT) matrix
 * to int8 q [N][K] (device) and its fp16 scales [N][K/128] (device, nullable)
 * for bit-exact checks. A ternary code 11 writes 0 to q and sets
 * QMV_ERR_CORRUPT in the device error word.
 */
int qmv_unpack(const qmv_desc* desc, const void* packed, int8_t* q, uint16_t* scales, void* stream);

/*
 * y[m][n] = sum_k W_hat[n][k] * x[m][k] for m < M, n < N, where W_hat = q * scale
 * of the packed ternary (qmv_run_ternary) or INT4 (qmv_run_int4) matrix.
 * M in 1..QMV_MAX_M, ldx >= K, ldy >= N (a QMV_TERNARY2_SPARSE desc in
 * qmv_run_ternary or qmv_run_batch: M in 1..8, the fp16-FMA kernel, and K must
 * fit shared memory in one piece). Every kernel decodes a zero code to an
 * exact 0, so an activation meeting a zero weight contributes nothing. The
 * tensor-core kernel multiplies the bf16 activations as given (exact products)
 * and sums in fp32. The fp16-FMA kernel (and the sparse kernel) scales each
 * activation row and chunk of K by a power of two into fp16, where every value
 * down to 2^-30 (ternary) or 2^-25 (INT4) of the chunk's largest magnitude is
 * exact, forms exact products and sums them in fp16 chains of 8 columns (at
 * most 3 * 2^-11 of the chain's sum of |terms|), then in fp32. Each row's
 * error stays within the library's bound
 * |y - y_exact| <= 2e-3 * sum_k |W_hat[n][k] x[m][k]|
 * (for the fp16-FMA kernel: for activations within that range).
 */
int qmv_run_ternary(const qmv_desc* desc, const void* w, const void* x_bf16, int M, int64_t ldx,
                    float* y, int64_t ldy, void* stream);
/*
 * A QMV_INT4_LUT desc in qmv_run_int4 or qmv_run_batch serves M = 1 only and
 * runs the same byte-lookup kernel with one table entry per column pair (256
 * code bytes per pair, q_lo x_2p + q_hi x_2p+1 in fp32).
 * A QMV_TERNARY2_LUT desc in qmv_run_ternary or qmv_run_batch serves M = 1
 * only (QMV_ERR_UNSUPPORTED otherwise; ldx and ldy are then unused) and runs
 * the byte-lookup kernel: per block of 128 columns it builds, in fp32, the
 * sum of q_i x_i over each column group of four for all 81 valid code bytes,
 * then adds one table entry per code byte and multiplies each block's sum by
 * its scale, all in fp32; y is written without atomics (deterministic). A code
 * byte holding a code 11 contributes 0. Small launches split each matrix's
 * blocks over a cluster of up to 8 CTAs.
 */
int qmv_run_int4(const qmv_desc* desc, const void* w, const void* x_bf16, int M, int64_t ldx,
                 float* y, int64_t ldy, void* stream);

/*
 * Several independent matvecs of one format and one M in a single persistent
 * launch (a whole decode stack's q/k/v/o/gate/up/down, or the q|k|v and
 * gate|up groups that share one x). 1 <= n_tasks <= QMV_MAX_BATCH. The tasks
 * must not write overlapping y ranges. The kernel choice follows the OR of the
 * descriptors' QMV_FLAG_PATH_* bits.
 */
int qmv_run_batch(int format, const qmv_task* tasks, int n_tasks, int M, void* stream);

/*
 * Cassandra offline transform on the host ("Cassandra", 3.2-3.3).
 * w_bf16: host [N][K] bf16 bits; calib_bf16: host [R][K] bf16 calibration
 * activations. Keeps the K/2 largest Wanda scores |w| * ||X[:,j]||_2 of each
 * row (float64; equal scores keep the lower column; NaN scores as +inf), splits
 * kept values into sign + 3 high mantissa bits and 4 low mantissa bits, ranks
 * exponents of the kept values by frequency (ties: smaller exponent first) and
 * writes each as a unary code. K must be a positive multiple of 32, N, R > 0.
 * With out == NULL only `desc` is filled (size query). With out != NULL,
 * out_capacity must be >= desc->total_bytes. out is host memory.
 */
int cass_pack_host(const uint16_t* w_bf16, int64_t N, int64_t K, const uint16_t* calib_bf16,
                   int64_t R, qmv_desc* desc, void* out, int64_t out_capacity);

/*
 * Cassandra-2 offline transform on the host ("Cassandra", 3.3, MX route): the
 * same Wanda selection as cass_pack_host, then the QMV_CASS_MX layout (see
 * qmv_desc). K must be a positive multiple of 64, N, R > 0. The layout depends
 * only on N and K (desc equals qmv_pack_desc(QMV_CASS_MX, N, K, 32)). With out
 * == NULL only `desc` is filled; otherwise out_capacity >= desc->total_bytes.
 * out is host memory.
 */
int cass_mx_pack_host(const uint16_t* w_bf16, int64_t N, int64_t K, const uint16_t* calib_bf16,
                      int64_t R, qmv_desc* desc, void* out, int64_t out_capacity);

/*
 * Online KV-cache encoder on the GPU ("Cassandra", 3.5: new K/V are pruned,
 * truncated and encoded as they are produced; 3.2: the KV cache is pruned by
 * per-token magnitude). kv: device bf16 [T][ld], one token's D values per row.
 * Keeps the D/2 largest |v| of each row (equal magnitudes: lower index first;
 * NaN as +inf), splits the kept values as cass_pack_host does, and writes each
 * exponent as a unary code of its rank in `codebook` (host, the 256 exponent
 * values in rank order, each once) into a fixed slot of slot_words 32-bit words
 * per row (rowstart[n] = n * slot_words, zero-filled after the codes). The
 * result is a QMV_CASS buffer (n_symbols 256) that cass_decode_draft and
 * cass_reconstruct read. D % 32 == 0, D <= 16384, slot_words a positive
 * multiple of 4. desc is filled on the host; with packed == NULL nothing runs
 * (size query), otherwise packed (device, capacity >= desc->total_bytes) is
 * written on `stream`. A row whose codes exceed its slot keeps the codes that
 * fit and records QMV_ERR_UNSUPPORTED in the device error word.
 */
int cass_kv_encode(const uint16_t* kv, int64_t T, int64_t D, int64_t ld, const uint8_t* codebook,
                   int64_t slot_words, qmv_desc* desc, void* packed, int64_t capacity, void* stream);

/*
 * Draft path ("Cassandra", 3.2 figure b): reads only the speculation sections
 * of the packed buffer (QMV_CASS: 0-4, QMV_CASS_MX: 0-3). Draft weight = S<<15 |
 * E<<7 | m_hi<<4 for kept values (low mantissa bits zero-filled; QMV_CASS_MX:
 * the sign and A >> 4 at the group exponent), +0 for pruned values.
 * y: device fp32 [M][ldy] or NULL; w_draft: device bf16 bits [N][K] or NULL
 * (materialised draft weights, for bit-exact checks). M in 1..8.
 * A unary rank beyond the codebook or a bitmap row without exactly K/2 kept
 * values sets QMV_ERR_CORRUPT.
 */
int cass_decode_draft(const qmv_desc* desc, const void* packed, const void* x_bf16, int M,
                      int64_t ldx, float* y, int64_t ldy, uint16_t* w_draft, void* stream);

/*
 * Target path ("Cassandra", 3.2 figure c): reads speculation and verification
 * data and rebuilds every original bf16 bit before the matvec (QMV_CASS_MX:
 * the MX target values, see qmv_desc). Same argument rules as
 * cass_decode_draft; w_out receives the reconstructed bf16 bits.
 */
int cass_reconstruct(const qmv_desc* desc, const void* packed, const void* x_bf16, int M,
                     int64_t ldx, float* y, int64_t ldy, uint16_t* w_out, void* stream);

/*
 * One draft-then-verify step of self-speculative decoding on one Cassandra
 * matrix ("Cassandra", section 2 and 3.2 figures b and c: draft tokens come from
 * the speculation data alone, then one target pass over speculation and
 * verification data checks the current token and every draft token at once).
 * Activation row 0 of x is the current token, rows 1..n_draft the draft tokens.
 * Issues, in stream order, n_draft draft matvecs at M = 1 (y_draft[d] = W_draft
 * x[d] for d < n_draft: draft token d + 1 is produced from row d) and then one
 * target matvec at M = n_draft + 1 (y_target[m] = W x[m], W the original
 * bf16 weights rebuilt bit for bit). x: device bf16 [n_draft + 1][ldx];
 * y_draft: device fp32 [n_draft][ldy]; y_target: device fp32
 * [n_draft + 1][ldy]; the two must not overlap. 1 <= n_draft <= 7 (the
 * "Nemotron 3.5 Bolt" drafts are 7 tokens long). QMV_CASS or QMV_CASS_MX.
 * Every argument is checked before the first launch; errors as
 * cass_decode_draft.
 */
int cass_speculate_step(const qmv_desc* desc, const void* packed, const void* x_bf16, int n_draft, int64_t ldx,
                        float* y_draft, float* y_target, int64_t ldy, void* stream);

/*
 * Mixture-of-experts decode over ternary SwiGLU experts ("Nemotron 3.5 Bolt",
 * expert top-K routing): per token, the top-k of E router logits (equal logits:
 * lower expert index first; -0 equals +0 and a NaN logit ranks as -inf), p = softmax
 * over the k selected logits (fp32), and
 *   y_t = sum_e p_{t,e} * W_down,e ( silu(W_gate,e x_t) * (W_up,e x_t) ).
 * Only the selected experts' packed weights are read.
 * experts: device; expert e's record starts at experts + e * expert_stride and
 * holds the packed [gate; up] matrix (2I x H, described by gateup_desc, rows
 * 0..I-1 gate and I..2I-1 up) followed, at byte offset down_off, by the packed
 * down matrix (H x I, down_desc). Both ternary, in one layout: QMV_TERNARY2
 * (row-group records; fp16-FMA expert kernels, one slot per active expert with
 * all its tokens) or QMV_TERNARY2_LUT (byte-lookup layout; the lookup kernel, one
 * task per (token, expert) pair, H and I multiples of 128; y is added into in a
 * run-dependent order, within the same bound). logits: device fp32 [M][E].
 * x_bf16: device [M][ldx]; y: device fp32 [M][ldy], overwritten.
 * workspace: device, >= moe_workspace_size(E, topk, M, H, I) bytes.
 * 1 <= topk <= 8, topk <= E <= 256, M in 1..8.
 */
size_t moe_workspace_size(int E, int topk, int M, int64_t H, int64_t I);
int moe_qmv_run(const qmv_desc* gateup_desc, const qmv_desc* down_desc, const void* experts,
                int64_t expert_stride, int64_t down_off, int E, const float* logits, int topk,
                const void* x_bf16, int M, int64_t ldx, float* y, int64_t ldy,
                void* workspace, size_t ws_bytes, void* stream);

/*
 * The same MoE decode as moe_qmv_run, for callers that cannot allocate device
 * memory themselves: for example a plugin inside a host application that owns
 * every device allocation, or a latency-critical loop that must not pay for
 * cudaMalloc. Instead of a caller workspace it uses one fixed scratch array of
 * QMV_MOE_STATIC_SCRATCH_BYTES bytes that lives in this library's own device
 * memory (every GPU that loads the library holds it until the process exits).
 * The pages have no counterpart to this entry point; it exists only for such
 * callers.
 *  - It allocates nothing and frees nothing. The first call on a device looks up
 *    the array's device address (cudaGetSymbolAddress) and keeps it; make that
 *    first call before any stream capture. The kept address belongs to the
 *    device's context: after cudaDeviceReset on that device do not call this
 *    entry point again in the same process.
 *  - A call whose scratch need (moe_workspace_size) exceeds the array is
 *    rejected with QMV_ERR_ARG before any launch.
 *  - All calls share the one array and it keeps the previous call's contents;
 *    each call rewrites everything it reads, so nothing needs clearing. Calls
 *    that overlap on the GPU (for example on two streams) race on the array:
 *    issue them in one stream order.
 * Other arguments, layouts and errors are those of moe_qmv_run.
 */
#define QMV_MOE_STATIC_SCRATCH_BYTES (2u * 1024u * 1024u)
int moe_qmv_run_static(const qmv_desc* gateup_desc, const qmv_desc* down_desc, const void* experts,
                       int64_t expert_stride, int64_t down_off, int E, const float* logits, int topk,
                       const void* x_bf16, int M, int64_t ldx, float* y, int64_t ldy, void* stream);

/*
 * Packed-weight files ("Ternary Bonsai 2", section 3.6: the packed indices,
 * scales and flags are exported as the file that inference loads). A file
 * holds named packed matrices of any format above, each with its qmv_desc and
 * a CRC-32 per section (reflected polynomial 0xEDB88320, as zip), behind a
 * versioned header whose own fields and entry table carry CRC-32s too; the byte
 * layout is described in the library source (file.cu). Tensors start on 4096-byte
 * boundaries. Host-side calls; only qmv_file_load touches the GPU.
 *
 * qmv_file_write: names[i] (NUL-terminated, < QMV_FILE_NAME_BYTES bytes,
 *   unique), descs[i] and buffers[i] (host, descs[i].total_bytes bytes) of n
 *   tensors; the descriptors' flags are stored as 0. Overwrites `path`.
 * qmv_file_open: maps the file read-only and checks magic, version, header and
 *   table CRCs and that every entry lies inside the file with a valid
 *   descriptor (QMV_ERR_CORRUPT otherwise; QMV_ERR_UNSUPPORTED for a newer
 *   version). *out is freed by qmv_file_close.
 * qmv_file_tensor: name (nullable, QMV_FILE_NAME_BYTES bytes) and descriptor
 *   (nullable) of tensor `index`; qmv_file_find: the index of a name, or
 *   QMV_ERR_ARG if absent.
 * qmv_file_load: checks the CRC of every section of tensor `index` on the host
 *   (QMV_ERR_CORRUPT on a mismatch, nothing copied), then copies the packed
 *   buffer into `dst` (device, caller-owned, >= desc.total_bytes bytes,
 *   16-byte aligned) on `stream`. When the call returns the source bytes are
 *   staged, so the file may be closed while the copy is in flight.
 * qmv_file_read_host: the same check, then a copy into host memory.
 * qmv_crc32: CRC-32 of n bytes continuing from `crc` (0 to start).
 */
#define QMV_FILE_NAME_BYTES 64
typedef struct qmv_file qmv_file;
int qmv_file_write(const char* path, int n, const char* const* names, const qmv_desc* descs,
                   const void* const* buffers);
int qmv_file_open(const char* path, qmv_file** out);
int qmv_file_count(const qmv_file* f);
int qmv_file_tensor(const qmv_file* f, int index, char* name, qmv_desc* desc);
int qmv_file_find(const qmv_file* f, const char* name);
int qmv_file_load(const qmv_file* f, int index, void* dst, int64_t capacity, void* stream);
int qmv_file_read_host(const qmv_file* f, int index, void* dst, int64_t capacity);
void qmv_file_close(qmv_file* f);
uint32_t qmv_crc32(const void* data, size_t n, uint32_t crc);

/*
 * Synchronize `stream`, then read and clear the current device's error word.
 * *device_code (nullable) receives 0 or a qmv_status the kernels recorded.
 * Returns QMV_ERR_CUDA if the synchronization failed, else the recorded status.
 */
int qmv_check_status(void* stream, int32_t* device_code);

/* Message for the calling thread's last failed call ("" if none). */
const char* qmv_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* QMV_H */
