/*
 * q4mm.h -- C ABI of libq4mm, the GB300 (sm_103a) Q4_0 quantized linear layer.
 *
 * The operation (rembed "Architecture", section "The pluggable kernel
 * interface": MatMul(dst, a, bT, m, k, n), C[m x n] = A[m x k] . B^T with
 * B^T stored [n x k] row-major, an nn.Linear weight as stored):
 *
 *     Y[t][j] = sum_c X[t][c] * W[j][c]        t < m, j < n, c < k
 *
 * W is held as GGUF Q4_0 blocks (the format of the Q4_0 GGUF files the golem
 * page runs, "Quickstart"): each block covers 32 consecutive weights of one
 * row and is 18 bytes, an IEEE binary16 scale d (little endian) followed by
 * qs[16]; byte i of qs holds weight i in its low nibble and weight i+16 in
 * its high nibble (goinfer ch. 10, "Kernels and backends", section "Layout,
 * concretely"); a weight is (q - 8) * d.
 *
 * One library call serves the three regimes the pages run the layer in:
 * decode (m = 1), continuous batching where several slots' tokens share one
 * read of the weights (golem, "Several conversations, one pass"; golem-server,
 * "Several conversations, in one pass"), and prompt reading, where wide
 * passes use tiled products ("Reading a prompt on the card": the mat-vec is
 * built up to sixteen columns, tiled products take over from thirty-two).
 *
 * Conventions for every entry point:
 *   - Pointers named W_packed, blocks, X, Y, X_slots, Y_slots, slot_ids and
 *     workspace are DEVICE pointers of the current CUDA device. The caller
 *     owns and allocates every buffer; nothing is freed by the library.
 *   - Work is enqueued on `stream` and the call returns without waiting.
 *     Argument errors are returned synchronously before anything is enqueued.
 *     A launch failure is returned as Q4_ERR_CUDA. A fault found by a kernel
 *     while it runs (a bounded wait that ran out) is recorded in a per-device
 *     status word that q4_last_device_status() reads once the stream has been
 *     synchronised.
 *   - There is no fallback: a device other than compute capability 10.3 is
 *     refused with Q4_ERR_UNSUPPORTED_DEVICE.
 *   - Results are bitwise identical from run to run for the same inputs and
 *     sizes (no floating-point atomics; split sums are added in a fixed
 *     order).
 */
#ifndef Q4MM_H
#define Q4MM_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st;
/* Same type as cudaStream_t; NULL is the legacy default stream. */
typedef struct CUstream_st *q4mm_stream_t;

#if defined(__GNUC__)
#define Q4MM_API __attribute__((visibility("default")))
#else
#define Q4MM_API
#endif

/* Status codes. */
#define Q4_OK 0
#define Q4_ERR_INVALID_ARG 1        /* null pointer, k % 32 != 0, n <= 0, k <= 0, m < 0, bad ld */
#define Q4_ERR_ALIGNMENT 2          /* a pointer or leading dimension breaks the alignment rule */
#define Q4_ERR_UNSUPPORTED_DEVICE 3 /* current device is not compute capability 10.3 (GB300) */
#define Q4_ERR_CUDA 4               /* a CUDA runtime call or kernel launch failed */
#define Q4_ERR_DEVICE_TIMEOUT 5     /* a kernel's bounded wait ran out (read by q4_last_device_status) */
#define Q4_ERR_WORKSPACE 6          /* workspace missing or smaller than q4_0_matmul_workspace_size() */
#define Q4_ERR_NO_MEMORY 7          /* the library could not allocate its own workspace */
#define Q4_ERR_IO 8                 /* a file could not be opened or read */
#define Q4_ERR_FORMAT 9             /* a file breaks the GGUF layout (q4_gguf_open) */
#define Q4_ERR_DEVICE_CHECK 10      /* checked build: a kernel found an index or offset out of range and
                                       skipped the access (read by q4_last_device_status) */

/*
 * Packed weight layout (what q4_0_pack writes). Repacking the blocks at load
 * for the kernels' access order is the pages' layout step (goinfer ch. 10,
 * "Making Go fast enough" and "Layout, concretely"; rembed "The pluggable
 * kernel interface": a second, packed-weight interface). The payload is the
 * same 18 bytes per block; only padding is added.
 *
 *   n is padded to a multiple of 128 rows (a group), k to a multiple of 64 (a
 *   pair of blocks). A record covers one group x one pair and is 4608 bytes:
 *     bytes    0..511   4 bytes per row r (at 4r): the fp16 scale bits of the
 *                       pair's first block (low half) and second block
 *                       (high half)
 *     bytes  512..2559  16 bytes per row r (at 512 + 16r): qs of the first block
 *     bytes 2560..4607  16 bytes per row r (at 2560 + 16r): qs of the second
 *   Records are ordered [group][pair], so a group's pairs are contiguous and a
 *   kernel thread that owns one row reads its share with three conflict-free
 *   shared-memory loads. Padding blocks have d = 0 and every nibble 8.
 */

/* Bytes of the packed form of an n x k Q4_0 matrix; 0 if n <= 0, k <= 0
 * or k % 32 != 0. */
Q4MM_API size_t q4_0_packed_size(int64_t n, int64_t k);

/* Repack GGUF Q4_0 blocks into the packed layout (run once, at load).
 *   W_packed: device, q4_0_packed_size(n, k) bytes, 16-byte aligned (written).
 *   blocks:   device, n * (k/32) blocks of 18 bytes, row-major [n][k/32],
 *             2-byte aligned (read).
 *   n, k:     rows (output features) and columns (input features), k % 32 == 0.
 * The two buffers must not overlap. Byte-exact: q4_0_unpack inverts it. */
Q4MM_API int q4_0_pack(void *W_packed, const void *blocks, int64_t n, int64_t k,
                       q4mm_stream_t stream);

/* Inverse of q4_0_pack: write the n x (k/32) GGUF blocks back out.
 *   blocks: device, n * (k/32) * 18 bytes, 2-byte aligned (written).
 *   W_packed: device, as written by q4_0_pack for the same n, k (read). */
Q4MM_API int q4_0_unpack(void *blocks, const void *W_packed, int64_t n, int64_t k,
                         q4mm_stream_t stream);

/* Bytes of device scratch q4_0_matmul_ws / q4_0_matmul_batched_slots_ws need
 * for these sizes: 0 for m <= 16 (decode needs none), the bf16 X image for
 * m > 16. */
Q4MM_API size_t q4_0_matmul_workspace_size(int64_t m, int64_t k, int64_t n);

/* Y[m x n] = X[m x k] . W^T, W given in packed form.
 *   W_packed: device, packed by q4_0_pack for (n, k), 16-byte aligned.
 *   X: device fp32 [m x k] row-major, 16-byte aligned.
 *   Y: device fp32 [m x n] row-major, overwritten (no accumulate); 4-byte aligned.
 *   m >= 0 (m == 0 does nothing), n >= 1, k >= 32, k % 32 == 0.
 * Precision (m <= 16, see q4_set_decode_kernel for which kernel runs):
 * the warp-MMA kernel forms each weight's (q - 8) exactly, scales each
 * 32-element block of an X row by a power of two and splits it into two fp16
 * terms (22 significant bits relative to the block's largest |x|), and
 * accumulates in fp32, applying d in fp32 per block; the CUDA-core kernel
 * uses (q - 8) exactly and X unrounded, in fp32; the tcgen05 kernel rounds
 * each weight (q - 8) * d once to fp16 (relative error <= 2^-11, scales |d|
 * <= 4096) and splits each X row, scaled by a power of two, into two fp16
 * terms. Each meets |Y - Y_exact| <= 1e-3 * B + 1e-5, B = sum_c |X[t][c] *
 * W[j][c]|. For m > 16 X is rounded to bf16 (nearest even), each weight is
 * the exact (q - 8) times d rounded to bf16, rounded to bf16 (relative error
 * <= 2^-8), and the tensor cores accumulate in fp32: |Y - Y_exact| <= 1e-2 *
 * B + 1e-4 (17..32 rows, with the default decode kernel, may instead run as
two decode calls of 16 rows and the rest, where that is estimated faster for
the layer; they then meet the decode bound). NaN and infinity in X propagate
as in IEEE arithmetic.
 * Scratch: this form uses a workspace the library allocates on the current
 * device, once per (device, stream), grown when a call needs more. A call
 * that has to grow it synchronises `stream` and is refused with
 * Q4_ERR_WORKSPACE while the stream is being captured; make one call of the
 * largest size before capturing. Use q4_0_matmul_ws to pass your own. */
Q4MM_API int q4_0_matmul(const void *W_packed, const float *X, float *Y,
                         int64_t m, int64_t k, int64_t n, q4mm_stream_t stream);

/* As q4_0_matmul with caller-owned scratch: `workspace` (device, 256-byte
 * aligned) of at least q4_0_matmul_workspace_size(m, k, n) bytes, which may be
 * NULL when that size is 0. The library never allocates in this form.
 * The workspace holds the bf16 image of X that the prefill path (m > 16)
 * builds; it needs no initialisation (each call writes what it reads), so
 * one workspace serves calls of any shape in turn. Calls that can run at the
 * same time need distinct workspaces. */
Q4MM_API int q4_0_matmul_ws(const void *W_packed, const float *X, float *Y,
                            int64_t m, int64_t k, int64_t n,
                            void *workspace, size_t workspace_bytes, q4mm_stream_t stream);

/* Expert-grouped product (a mixture of experts): X's rows are grouped by
 * expert, rows offsets[e] .. offsets[e+1] - 1 going to expert e, and
 * Y[r] = X[r] . W_e^T for those rows (golem-server, "Several conversations,
 * in one pass", on mixture layers: the weights an expert contributes are read
 * once for the columns routed to it). Each expert's weights are read once for
 * its rows (twice for 17..32 rows): experts with up to 32 rows run the decode
 * mat-vec in pieces of at most 16 rows, pieces of the same mat-vec instance
 * (1, 2, 4, 8 or 16 token columns) sharing one launch per set of up to 32 (a
 * thread-block cluster per 128-row group of a piece); larger groups run the
 * tensor-core GEMM one expert at a time (the switch at 32 rows is measured on
 * GB300: below it the pieces are faster than the GEMM). Each piece or group
 * has q4_0_matmul's precision for its size.
 *   W_packed: host array of n_experts device pointers, each packed by
 *   q4_0_pack for (n, k), 16-byte aligned (an expert with no rows may be
 *   NULL).
 *   offsets: host array of n_experts + 1 row offsets, offsets[0] = 0,
 *   non-decreasing; the row count is offsets[n_experts].
 *   X: device fp32 [rows x k], 16-byte aligned; Y: device fp32 [rows x n],
 *   overwritten, 4-byte aligned.
 * The arguments are checked before anything is launched; if a later group
 * is refused (its plan, or the library workspace while a stream is being
 * captured), the groups before it have been written. Scratch: as
 * q4_0_matmul (the library's workspace, for groups of more than 32 rows). */
Q4MM_API int q4_0_matmul_experts(const void *const *W_packed, int64_t n_experts, const int64_t *offsets,
                                 const float *X, float *Y, int64_t k, int64_t n, q4mm_stream_t stream);

/* W4A8: Y[m x n] = X[m x k] . W^T with X coded to int8 first, so that every
 * block's dot product is an integer one. The pages name the integer dot
 * product (goinfer ch. 10, "Which kernel runs is a runtime decision": the
 * canonical quantized dot of integer-dot hardware; rembed "Architecture",
 * "int8 quantization": activations quantised, integer products bit-exact
 * against an integer reference) but print no coding rule; the one used:
 * per 32-element block of an X row, amax = max |x|, scale s = amax / 127 and
 * code c = round-half-even(x * (127 / amax)), all in fp32 (one IEEE quotient
 * or product each), so |c| <= 127; a block with amax = 0 has codes 0 and
 * s = 0. Then Y[t][j] = sum_b d(j,b) * s(t,b) * sum_i (q - 8) * c: each block's
 * integer sum is exact (fp16 operands, fp32 accumulation of integers below
 * 2^24), d * s and the sum over blocks are fp32, so |Y - Y_w4a8| <= 4e-5 * B8
 * + 1e-6 against the fp64 value, B8 = sum_b |d s sum_i (q - 8) c|. A row of X
 * holding a NaN or an infinity gives NaN in every output of that row.
 *   W_packed: device, packed by q4_0_pack for (n, k), 16-byte aligned.
 *   X: device fp32 [m x k] row-major, 16-byte aligned; Y: device fp32
 *   [m x n] row-major, overwritten, 4-byte aligned.
 *   0 <= m <= 16 (m == 0 does nothing; larger m is refused with
 *   Q4_ERR_INVALID_ARG), n >= 1, k >= 32, k % 32 == 0.
 * Runs in the whole-record decode kernel, eight tokens per MMA column tile;
 * needs no scratch and allocates nothing. */
Q4MM_API int q4_0_matmul_w4a8(const void *W_packed, const float *X, float *Y,
                              int64_t m, int64_t k, int64_t n, q4mm_stream_t stream);

/* Per-output-channel int8 weights (rembed "Architecture", "int8 quantization",
 * the weight-only form: dense weights quantised once at load to symmetric
 * int8 with one scale per output channel, dequantised in registers, the
 * channel's scale applied once in the epilogue).
 *
 * Bytes the packed form of an n x k fp32 weight matrix occupies: records of
 * 128 rows x 64 columns of codes, then one fp32 scale per row (rows padded to
 * a multiple of 128). 0 for invalid sizes (n < 1, k < 32, k % 32 != 0). */
Q4MM_API size_t q4_w8_packed_size(int64_t n, int64_t k);

/* Quantise W [n x k] (device fp32, row-major, 16-byte aligned, finite) into
 * W8_packed (device, q4_w8_packed_size bytes, 16-byte aligned; written).
 * Row j, every step one IEEE fp32 operation: amax = max |w|, scale
 * s = amax / 127, code c = round-half-even(w * (127 / amax)) (|c| <= 127); a
 * row with amax = 0 has codes 0 and s = 0. Enqueued on `stream`. */
Q4MM_API int q4_w8_quantize(void *W8_packed, const float *W, int64_t n, int64_t k, q4mm_stream_t stream);

/* The codes (device int8 [n x k], row-major, 4-byte aligned) and scales
 * (device fp32 [n]) held in W8_packed: the inverse of q4_w8_quantize's
 * layout, for checking it. */
Q4MM_API int q4_w8_unpack(int8_t *codes, float *scales, const void *W8_packed, int64_t n, int64_t k,
                          q4mm_stream_t stream);

/* Y[m x n] = X[m x k] . W8^T with W8[j][c] = s_j * code[j][c]: the codes are
 * exact in fp16 and X is split per 64 columns, scaled by a power of two, into
 * fp16 hi + lo (22 significant bits relative to those columns' largest |x|);
 * the tensor cores accumulate in fp32 and s_j scales each output once:
 * |Y - Y_exact| <= 1e-3 * B + 1e-5, B = sum_c |X[t][c] * s_j * code[j][c]|.
 * NaN and infinity in X propagate.
 *   W8_packed: as written by q4_w8_quantize for (n, k); X: device fp32 [m x k]
 *   row-major, 16-byte aligned; Y: device fp32 [m x n], overwritten, 4-byte
 *   aligned. m >= 0 (m == 0 does nothing), n >= 1, k >= 32, k % 32 == 0.
 * Runs the decode mat-vec for up to 16 rows of X at a time (a larger m is
 * taken in launches of 16 rows, or of 8 or 4 where a long k leaves no room
 * for 16); needs no scratch and allocates nothing. */
Q4MM_API int q4_w8_matmul(const void *W8_packed, const float *X, float *Y, int64_t m, int64_t k, int64_t n,
                          q4mm_stream_t stream);

/* Size of the library's fixed scratch array used by q4_0_matmul_static_scratch. */
#define Q4_STATIC_SCRATCH_BYTES (8u << 20)

/* As q4_0_matmul, but with no allocation of any kind: the scratch is a fixed
 * array of Q4_STATIC_SCRATCH_BYTES (8 MiB) in the library's device memory,
 * one per device. The pages have no counterpart; this form exists for
 * callers that must not allocate device memory. Only m > 16 uses scratch.
 *   Limit: shapes with q4_0_matmul_workspace_size(m, k, n) above
 *   Q4_STATIC_SCRATCH_BYTES are refused with Q4_ERR_WORKSPACE before anything
 *   is launched (m = 540, n = 9728, k = 2560 needs about 3 MiB).
 *   Set-up: the first call on a device, with that device current, looks up
 *   the array's address (cudaGetSymbolAddress, return code checked). Make
 *   that first call before any stream capture; later calls only enqueue work
 *   on `stream`. The array needs no zeroing: each call writes the part it
 *   reads.
 *   Races: every call on a device shares the one array, so calls that can
 *   overlap (other streams, other threads) race; calls in one stream are
 *   ordered.
 * Arguments, precision and status codes as q4_0_matmul. */
Q4MM_API int q4_0_matmul_static_scratch(const void *W_packed, const float *X, float *Y,
                                        int64_t m, int64_t k, int64_t n, q4mm_stream_t stream);

/* Continuous batching: m active slots share one read of the weights.
 * For i < m, row slot_ids[i] of X_slots produces row slot_ids[i] of Y_slots;
 * every other row of Y_slots is left untouched. Equivalent to gathering the
 * rows, q4_0_matmul, and scattering the results, with no extra copies.
 *   X_slots: device fp32, row r at X_slots + r * ldx; ldx >= k, ldx % 4 == 0,
 *            X_slots 16-byte aligned.
 *   slot_ids: device int32[m], distinct, each in [0, number of slot rows).
 *            Distinctness and range are the caller's contract (not checked on
 *            the device; a repeated id makes the written row undefined).
 *   Y_slots: device fp32, row r at Y_slots + r * ldy; ldy >= n.
 * Same precision and scratch rules as q4_0_matmul. */
Q4MM_API int q4_0_matmul_batched_slots(const void *W_packed, const float *X_slots, int64_t ldx,
                                       const int32_t *slot_ids, int64_t m,
                                       float *Y_slots, int64_t ldy,
                                       int64_t k, int64_t n, q4mm_stream_t stream);

/* As q4_0_matmul_batched_slots with caller-owned scratch (see q4_0_matmul_ws). */
Q4MM_API int q4_0_matmul_batched_slots_ws(const void *W_packed, const float *X_slots, int64_t ldx,
                                          const int32_t *slot_ids, int64_t m,
                                          float *Y_slots, int64_t ldy,
                                          int64_t k, int64_t n,
                                          void *workspace, size_t workspace_bytes,
                                          q4mm_stream_t stream);

/* Human-readable name of a status code (static string, never NULL). */
Q4MM_API const char *q4_status_string(int status);

/* Device status word of the current device: Q4_OK, Q4_ERR_DEVICE_TIMEOUT if
 * a kernel's bounded wait ran out, or Q4_ERR_DEVICE_CHECK (checked build
 * only) if a kernel's range check failed, since the word was last cleared
 * (the first such event is kept). Synchronises the device. clear != 0 resets
 * the word to Q4_OK. */
Q4MM_API int q4_last_device_status(int clear);

/* How this library was built: bit 0 set for the checked build (-DQ4MM_CHECKED:
 * the decode mat-vec checks its shared-memory layout against the launch's
 * size, every weight record it copies against the layer's records and
 * every slot row against the ring, and on a failed check records
 * Q4_ERR_DEVICE_CHECK in the status word and skips the access instead of
 * faulting), bit 1 for the event-trace build (-DQ4MM_TRACE). */
Q4MM_API int q4_build_flags(void);

/* Limit, in nanoseconds, on each device-side wait of the library's kernels
 * (default 2e9). Applies to launches made after the call, on every device.
 * A wait that runs out sets Q4_ERR_DEVICE_TIMEOUT in the device status word
 * and the kernel returns without its result. The decode mat-vec (the default
 * path for m <= 16) then still waits, for at least 0.2 s, for the transfers
 * already issued into its own shared memory, so any limit >= 1 is safe there;
 * the other kernels take the limit as given for every wait and need one well
 * above their transfers' latency (>= 1 ms). */
Q4MM_API int q4_set_wait_limit_ns(uint64_t ns);

/* Declare packed weights read-only while matmuls run (default: not declared).
 * When enabled, the matmul kernels (the decode kernel, and the prefill GEMM)
 * start streaming W_packed before the kernels that precede them in the
 * stream have finished, overlapping the two (programmatic dependent launch);
 * X, Y and the workspace are still read only after those kernels complete.
 * Enable it only if no kernel writes a W_packed immediately before a matmul
 * that reads it in the same stream (after q4_0_pack, synchronise or record an
 * event before the first matmul). Applies to launches made after the call. */
Q4MM_API int q4_set_weight_prefetch(int enable);

/* Decode kernels (m <= 16). Every one meets the decode tolerance; which one
 * runs is a performance choice. The pages bound decode by the weight read
 * (golem, "Qwen3.8 drafts its own next token"), so the kernels differ in how
 * few instructions they spend per weight byte:
 *   Q4_DECODE_AUTO       the library's choice for each call (default):
 *                        record MMA for m <= 4, and for m <= 8 on layers of
 *                        at most two 128-row groups per SM; warp-MMA
 *                        otherwise;
 *   Q4_DECODE_WARP_MMA   CUDA cores dequantise to exact fp16 (q - 8), the
 *                        warp-level MMA (mma.sync) multiplies by X split into
 *                        fp16 hi + lo, d is applied in fp32 per block;
 *   Q4_DECODE_CUDA_CORE  exact fp32 (q - 8), fp32 X, fp32 FMAs (m <= 4; wider
 *                        calls take Q4_DECODE_WARP_MMA);
 *   Q4_DECODE_TCGEN05    (q - 8) * d rounded to fp16 into tensor memory, X
 *                        split into fp16 hi + lo, tcgen05.mma;
 *   Q4_DECODE_RECORD_MMA each warp takes whole records: exact fp16 (q - 8)
 *                        times X split per block into fp16 hi + lo on the
 *                        warp-level MMA, d applied in fp32 per block (m <= 16);
 *   Q4_DECODE_MATVEC     the mat-vec: bf16 128 + q times X split per block
 *                        into fixed-point bf16 hi + lo on the warp-level MMA,
 *                        the accumulator starting at the bias correction so
 *                        that every block dot product is exact; four blocks
 *                        per accumulator tile at m = 1 (m <= 16).
 * The setting is kept per process and applies to launches made after the
 * call. Other values are refused with Q4_ERR_INVALID_ARG. */
#define Q4_DECODE_AUTO 0
#define Q4_DECODE_WARP_MMA 1
#define Q4_DECODE_CUDA_CORE 2
#define Q4_DECODE_TCGEN05 3
#define Q4_DECODE_RECORD_MMA 4
#define Q4_DECODE_MATVEC 5
Q4MM_API int q4_set_decode_kernel(int kind);

/* Profiling builds only (compiled with -DQ4MM_TRACE): kernels launched after
 * the call write 16-byte event records {globaltimer ns, event << 16 | warp
 * << 8 | lane, argument} for the CTA with blockIdx.x == cta into `buffer`
 * (device memory, 16-byte aligned, zeroed by the caller), split into 96
 * equal regions, one per recording thread (lanes 0..3 of warps 0..23); a
 * zero timestamp ends a region. NULL switches tracing off. Normal builds
 * return Q4_ERR_INVALID_ARG. */
Q4MM_API int q4_debug_set_trace(void *buffer, size_t bytes, uint32_t cta);

/* Self-test of the bounded-wait path: launches one block that waits on a
 * barrier nothing ever completes, for at most limit_ns nanoseconds, then
 * records Q4_ERR_DEVICE_TIMEOUT in the device status word and returns. */
Q4MM_API int q4_selftest_wait_timeout(uint64_t limit_ns, q4mm_stream_t stream);

/* ------------------------------------------------------------- GGUF --
 * A reader of GGUF files in front of q4_0_pack (host code, no device work).
 * "Go AI Inference: What is Inference?", section "GGUF: The Whole Model in
 * One File": a header (magic GGUF, version, tensor and metadata counts),
 * typed key-value metadata, tensor descriptors (name, shape, type, offset)
 * and the data blob; section "The blob: getting the weights into memory":
 * the loader parses the header, metadata and descriptors first, then places
 * each tensor's bytes. Field widths and type codes follow GGUF versions 2
 * and 3 as ggml writes them (little endian). A Q4_0 tensor (type 2) of
 * shape (k, n) (innermost first) holds the [n][k/32] 18-byte blocks that
 * q4_0_pack takes: read it with q4_gguf_read_tensor, copy it to the device,
 * pack it once. */
typedef struct q4_gguf q4_gguf;

/* Parse a file's header, metadata and tensor descriptors; no tensor data is
 * read. Every size is checked against the file: a file that breaks the
 * layout (bad magic, version other than 2 or 3, a string, array or tensor
 * reaching past the end, a descriptor offset not a multiple of
 * general.alignment, an array of arrays, more than 4 dimensions) gives
 * Q4_ERR_FORMAT; a file that cannot be read,
 * Q4_ERR_IO. On success *out owns the parsed file; release it with
 * q4_gguf_close. */
Q4MM_API int q4_gguf_open(const char *path, q4_gguf **out);
Q4MM_API void q4_gguf_close(q4_gguf *g);
/* Number of tensor descriptors (-1 for a null handle). */
Q4MM_API int64_t q4_gguf_tensor_count(const q4_gguf *g);
/* Index of the tensor called `name`, or -1. */
Q4MM_API int64_t q4_gguf_find_tensor(const q4_gguf *g, const char *name);
/* Descriptor of tensor `index`: name (owned by g), type, number of dims,
 * dims[4] (innermost first, unused ones 1), absolute byte offset of its data
 * in the file and its byte size (0 when the type's size is not one this
 * reader knows: f32, f16, Q4_0, Q8_0). Any output pointer may be NULL. */
Q4MM_API int q4_gguf_tensor_info(const q4_gguf *g, int64_t index, const char **name, int *type,
                                 int *n_dims, int64_t *dims, uint64_t *file_offset, uint64_t *bytes);
/* Read tensor `index`'s bytes into host memory of at least its byte size
 * (Q4_ERR_INVALID_ARG if smaller, or if the size is unknown). */
Q4MM_API int q4_gguf_read_tensor(const q4_gguf *g, int64_t index, void *host_dst, uint64_t dst_bytes);
/* A metadata value by key: an integer or bool scalar, or a string (owned by
 * g). Q4_ERR_INVALID_ARG when the key is absent or of another type. */
Q4MM_API int q4_gguf_get_int(const q4_gguf *g, const char *key, int64_t *value);
Q4MM_API int q4_gguf_get_string(const q4_gguf *g, const char *key, const char **value);

#ifdef __cplusplus
}
#endif

#endif /* Q4MM_H */
