/*
 * qr.h -- C ABI of libqr.so, a GB300 (sm_103a) implementation of the
 * quick-allreduce data path: a low-granularity block quantize/dequantize
 * codec and a one- and two-stage allreduce in which the W tensor-parallel
 * ranks are emulated as W fp16/bf16 buffers in one GPU's memory.
 *
 * Sources (web pages):
 *   vLLM PR #18473, "Integrate quick allreduce and select the best allreduce
 *     implementation": opening description (1stage f16; 2stage f16, fp8,
 *     Q8, Q6, Q4) and the tp2 kernel timing table.
 *   vLLM PR #16804, "Add quickreduce as alternative to custom allreduce":
 *     opening description (int4/int8, symmetric and asymmetric) and review
 *     discussion (one shot for small buffers, two shot for larger ones).
 *   vLLM API docs, "vllm.distributed.device_communicators.quick_all_reduce":
 *     QuickReduceRegime (FP=0, INT8=1, INT6=2, INT4=3), _SUPPORTED_DTYPES
 *     (float16, bfloat16), _SUPPORTED_WORLD_SIZES (2, 4, 8),
 *     should_quick_allreduce (input byte size a multiple of 16) and
 *     quick_all_reduce (out-of-place; ops.qr_all_reduce(..., level, ...)).
 *
 * Codec.  A message of n elements is cut into nb = ceil(n/32) blocks of 32.
 * Each block gets an fp16 scale s (and, for the asymmetric formats, an fp16
 * zero-point z) and 32 b-bit codes:
 *   symmetric  Q8/Q6/Q4 (b = 8/6/4): s = h(max|x| / Qmax), Qmax = 2^(b-1)-1,
 *              q = clamp(rne(x * (1/s)), -Qmax, Qmax), decoded as q*s;
 *   asymmetric Q8A/Q4A (b = 8/4):    s = h((max x - min x) / (2^b - 1)),
 *              z = h(min x), q = clamp(rne((x - z) * (1/s)), 0, 2^b - 1),
 *              decoded as q*s + z;
 *   FP8 (e4m3fn codes):              s = h(max|x| / 448),
 *              q = e4m3(x * (1/s)) rounded to nearest even and saturated,
 *              decoded as e4m3(q)*s;
 *   FP:        passthrough, no codes.
 * h() rounds binary32 to fp16 to nearest even and saturates at +-65504; all
 * arithmetic is binary32, round-to-nearest-even; a block whose scale
 * rounds to 0 gets all-zero codes.  The final block of a message whose n is
 * not a multiple of 32 takes its statistics over its valid elements; its
 * pad codes are 0.
 *
 * Encoded message layout (for qr_quantize's enc and qr_allreduce_emulated's
 * wire), structure of arrays:
 *   codes [nb][32*b/8 bytes]   code i of a block occupies bits [b*i, b*i+b)
 *                              of the block's little-endian bit stream;
 *                              symmetric codes are b-bit two's complement
 *   scales[nb]  fp16
 *   zps   [nb]  fp16           (asymmetric formats only)
 * For QR_FP the encoded message is the n values themselves (n*2 bytes).
 *
 * Conventions for every call:
 *   - All buffers are caller-owned DEVICE memory on the current device, and
 *     must be 16-byte aligned (qr_allreduce_host alone takes host buffers).
 *     The library allocates no memory.
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL = the legacy
 *     default stream).  QR_OK means the launch was accepted; a failed launch
 *     returns QR_ERR_CUDA.  Nothing synchronises the device.
 *   - Kernels are launched with programmatic stream serialization: each may
 *     become resident while the previous kernel on the stream drains, and
 *     waits for that kernel's completion before touching memory.  Each also
 *     lets the next kernel be scheduled early, so a kernel the caller
 *     launches after a call WITH that same attribute must call
 *     cudaGridDependencySynchronize() before reading the call's outputs (the
 *     general rule for programmatic dependent launch); ordinary launches,
 *     copies and events see the usual stream order.
 *   - n == 0 is a valid empty message: nothing is launched and pointers may
 *     be NULL.
 *   - Errors are reported by the return value only; no call aborts or
 *     prints.
 */
#ifndef QR_H
#define QR_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Message dtypes (_SUPPORTED_DTYPES on the quick_all_reduce API page).
 * QR_BF16_AS_F16 (qr_allreduce_emulated only): bf16 messages, processed the
 * way the bf16 -> fp16 cast option of init_quick_all_reduce on that page
 * describes -- each input rounded to fp16 (nearest even; values beyond
 * +-65504 become infinities, outside the contract), the fp16 allreduce run,
 * its fp16 result rounded to bf16 for `out`; the payload in `wire` is the
 * fp16 run's.  The other entry points reject it with QR_ERR_DTYPE. */
typedef enum { QR_F16 = 0, QR_BF16 = 1, QR_BF16_AS_F16 = 2 } qr_dtype;

/* Formats.  0..3 are QuickReduceRegime's values (FP, INT8, INT6, INT4) from
 * the quick_all_reduce API page; 4 is the "2stage f8" format of vLLM PR
 * #18473; 5 and 6 are the asymmetric int8/int4 formats of vLLM PR #16804. */
typedef enum {
  QR_FP = 0, QR_Q8 = 1, QR_Q6 = 2, QR_Q4 = 3,
  QR_FP8 = 4, QR_Q8_ASYM = 5, QR_Q4_ASYM = 6
} qr_format;

typedef enum {
  QR_OK = 0,
  QR_ERR_NULL = 1,    /* a required pointer is NULL (n > 0)                   */
  QR_ERR_DTYPE = 2,   /* dtype is not fp16 or bf16                            */
  QR_ERR_FORMAT = 3,  /* unknown format                                       */
  QR_ERR_WORLD = 4,   /* W not in {1, 2, 4, 8}                                */
  QR_ERR_STAGES = 5,  /* stages not in {1, 2}, or a wire buffer with stages 1 */
  QR_ERR_SIZE = 6,    /* n*2 bytes is not a multiple of 16, or n too large    */
  QR_ERR_ALIGN = 7,   /* a pointer is not 16-byte aligned                     */
  QR_ERR_OVERLAP = 8, /* an output buffer overlaps an input or another output */
  QR_ERR_CUDA = 9,    /* the CUDA runtime reported an error                   */
  QR_ERR_DEVICE = 10, /* a kernel gave up waiting (see qr_device_error)      */
  QR_ERR_SCRATCH = 11, /* qr_allreduce_staged_noalloc: the message needs more
                          stage-1 space than QR_NOALLOC_SCRATCH_BYTES        */
  QR_ERR_PATH = 12     /* qr_set_kernel_path: not one of the qr_path values   */
} qr_status;

/* Largest n accepted (elements per message): 2^36. */
#define QR_MAX_ELEMS ((uint64_t)1 << 36)

/* Bytes of one encoded message of n elements in format fmt:
 * nb*(32*b/8 + 2) for symmetric and FP8, nb*(32*b/8 + 4) for asymmetric,
 * n*2 for QR_FP; 0 for an unknown format.  Host only, no CUDA call. */
size_t qr_encoded_bytes(qr_format fmt, size_t n);

/* Encode one message (the codec's quantize step; the sender side of
 * "2stage ... Q8/Q6/Q4" in vLLM PR #18473).
 *   in   device, n values of dtype dt, 16-byte aligned, read only
 *   enc  device, qr_encoded_bytes(fmt, n) bytes, 16-byte aligned, written
 * enc must not overlap in. */
qr_status qr_quantize(qr_dtype dt, qr_format fmt, const void *in, size_t n,
                      void *enc, void *stream);

/* Decode one encoded message back to n values of dtype dt (the receiver
 * side of the codec).
 *   enc  device, qr_encoded_bytes(fmt, n) bytes, 16-byte aligned, read only
 *   out  device, n values of dtype dt, 16-byte aligned, written
 * out must not overlap enc. */
qr_status qr_dequantize(qr_dtype dt, qr_format fmt, const void *enc, size_t n,
                        void *out, void *stream);

/* Emulated quick allreduce of W messages (quick_all_reduce on the API page:
 * out-of-place, one call per allreduce; "1stage" and "2stage" of vLLM PR
 * #18473).  For every 32-element block, in this order:
 *   1. each rank's block is widened to binary32;
 *   2. stage 1 (reduce-scatter): for a quantized format every rank's block
 *      goes through the codec, xhat_r = decode(encode(x_r)); FP sends x_r;
 *   3. acc = xhat_0 + xhat_1 + ... + xhat_{W-1}, binary32, in rank order;
 *   4. stages == 2 (all-gather): a quantized format requantizes acc and
 *      every rank decodes the requantized block; FP rounds acc to dtype;
 *      stages == 1: acc is used as is (the one-shot variant: every rank
 *      reads every other rank's stage-1 data);
 *   5. out = the result rounded to dtype (round to nearest even).
 * The result is identical on all emulated ranks, so one copy is written.
 *   W       number of emulated ranks, 1, 2, 4 or 8 (1 = identity check)
 *   inputs  HOST array of W device pointers, each n values of dtype dt,
 *           16-byte aligned, read only (the array is read during the call)
 *   out     device, n values of dtype dt, 16-byte aligned, written
 *   wire    optional device buffer of qr_encoded_bytes(fmt, n) bytes that
 *           receives the stage-2 payload (the requantized blocks; for QR_FP
 *           the dtype-rounded sums); NULL to skip; must be NULL when
 *           stages == 1
 * out and wire must not overlap any input or each other. */
qr_status qr_allreduce_emulated(int W, qr_dtype dt, qr_format fmt, int stages,
                                const void *const *inputs, size_t n,
                                void *out, void *wire, void *stream);

/* Bytes of the stage-1 exchange buffer qr_allreduce_staged needs: W x W
 * slots, slot (j, r) holding rank r's chunk for owner j, with
 * chunk_nb = ceil(nb / W) blocks per owner, each slot an encoded
 * sub-message of chunk_nb blocks (codes | scales | zps; FP: the values)
 * padded to 16 bytes.  0 for an invalid W or format.  Host only. */
size_t qr_stage1_bytes(int W, qr_format fmt, size_t n);

/* The two-stage allreduce with its stage-1 exchange materialised, the
 * three-kernel structure a real multi-GPU quick allreduce has ("2stage" of
 * vLLM PR #18473): (1) each rank encodes its message and writes chunk j's
 * blocks into owner j's slot of `stage1` (reduce-scatter); (2) each owner
 * decodes its W slots, sums in rank order in binary32 and requantizes into
 * `wire` (the all-gather payload, same layout as qr_allreduce_emulated's);
 * (3) `wire` is decoded into `out`.  out and wire are bit-identical to
 * qr_allreduce_emulated(W, dt, fmt, 2, ...); only the memory traffic and
 * the number of launches differ.
 *   stage1  device, qr_stage1_bytes(W, fmt, n) bytes, 16-byte aligned,
 *           caller-owned scratch (contents on return: the stage-1 slots)
 *   wire    device, qr_encoded_bytes(fmt, n) bytes, required
 * All buffers 16-byte aligned; outputs must not overlap inputs or each
 * other.  Asynchronous on `stream` (three launches). */
qr_status qr_allreduce_staged(int W, qr_dtype dt, qr_format fmt,
                              const void *const *inputs, size_t n, void *out,
                              void *wire, void *stage1, void *stream);

/* qr_allreduce_staged without the caller's stage-1 buffer, for callers that
 * cannot allocate device memory: code that runs while a CUDA graph is being
 * captured, a plugin or callback that only receives its input and output
 * pointers and must not bypass its host framework's allocator, or a path
 * where cudaMalloc/cudaFree (and cudaFree's device synchronisation) are not
 * allowed.  The source pages have no counterpart: it exists for those
 * callers.
 *
 * The stage-1 buffer is a fixed device array inside this library of
 * QR_NOALLOC_SCRATCH_BYTES (16 MiB); every GPU on which the library is used
 * keeps it until the process exits.  Messages whose qr_stage1_bytes(W, fmt,
 * n) exceeds it are rejected with QR_ERR_SCRATCH (e.g. W=2 fp16 Q8 allows
 * about 7.8M elements per rank).  Nothing is allocated by the call.
 *
 * The first call on each device looks up the array's device address
 * (cudaGetSymbolAddress) and keeps it; make that first call before any
 * stream capture.  All calls share the one array: two calls whose work
 * overlaps on the GPU (different streams, no ordering between them) race on
 * it and their results are undefined; calls ordered on one stream are fine.
 * Nothing in the array needs to start at zero: stage 1 writes every byte the
 * owners read, whatever a previous call left there.
 * Arguments, results and other errors as qr_allreduce_staged. */
#define QR_NOALLOC_SCRATCH_BYTES ((size_t)16 << 20)
qr_status qr_allreduce_staged_noalloc(int W, qr_dtype dt, qr_format fmt,
                                      const void *const *inputs, size_t n,
                                      void *out, void *wire, void *stream);

/* Bytes of device workspace that qr_allreduce_host needs for W ranks, format
 * fmt and chunks of chunk_elems elements: two chunk buffers, each holding W
 * input chunks, the output chunk and the chunk's stage-2 payload, every
 * region padded to 256 bytes.  0 for an invalid W or fmt, or a chunk_elems
 * that is 0 or not a multiple of 32.  Host only, no CUDA call. */
size_t qr_host_workspace_bytes(int W, qr_format fmt, size_t chunk_elems);

/* qr_allreduce_emulated on HOST buffers (the quick_all_reduce call of the
 * vLLM quick_all_reduce page with its tensors in host memory): the W input
 * messages are read from host memory and the output (and optional stage-2
 * payload) written to host memory.  No counterpart on the pages, which work
 * on device tensors only; results are bit-identical to qr_allreduce_emulated
 * on device copies of the same inputs, because the method is defined block
 * by block.
 *
 * The message is processed in chunks of chunk_elems elements (a multiple of
 * 32; the last chunk may be shorter), double-buffered in `workspace`: the
 * copy-in of chunk i+1, the kernel on chunk i and the copy-out of chunk i-1
 * run at the same time on the two copy directions and the SMs.
 *   host_inputs  host array of W host pointers, n values of dtype dt each,
 *                read only; any alignment
 *   host_out     host, n values of dtype dt, written
 *   host_wire    host, qr_encoded_bytes(fmt, n) bytes in the layout of
 *                qr_allreduce_emulated's wire, written; or NULL.  Must be NULL
 *                when stages == 1
 *   workspace    device, at least qr_host_workspace_bytes(W, fmt,
 *                chunk_elems) bytes (workspace_bytes says how many), 16-byte
 *                aligned, owned by the caller; no other work may use it until
 *                this call's work on `stream` has completed
 * Host buffers should be page-locked (cudaHostAlloc or cudaHostRegister):
 * copies from or to pageable memory are correct but do not overlap.
 * Ordering: everything is ordered after prior work on `stream`, and work
 * later enqueued on `stream` runs after all of it, the last copy-out
 * included; the host buffers may be read or reused from then on.  The copies
 * run on two streams that the library creates per device on first use and
 * keeps; calls on one device enqueue one at a time (a mutex).  Not meant
 * for CUDA graph capture (use qr_allreduce_emulated inside graphs).
 * Errors: as qr_allreduce_emulated, plus QR_ERR_SIZE for a bad chunk_elems
 * or too small a workspace, QR_ERR_OVERLAP for host buffers that overlap;
 * QR_ERR_CUDA if a copy or a launch is refused (work enqueued before the
 * failure still runs). */
qr_status qr_allreduce_host(int W, qr_dtype dt, qr_format fmt, int stages,
                            const void *const *host_inputs, size_t n,
                            void *host_out, void *host_wire, void *workspace,
                            size_t workspace_bytes, size_t chunk_elems,
                            void *stream);

/* Kernel-path selection.  Every qr_quantize and qr_allreduce_emulated call is
 * served by one of three kernel paths that compute identical bits:
 *   QR_PATH_DIRECT           single-pass kernels with one memory round trip
 *                            (lowest latency): four lanes per block, or one
 *                            thread per block for qr_quantize and for the W=2
 *                            and W=4 calls of the integer formats from 3M / 4M
 *                            elements per rank;
 *   QR_PATH_PIPELINE_NARROW  the persistent bulk-copy pipeline with 8 KiB tiles
 *                            (mid-size messages: a shorter first fill and
 *                            last round);
 *   QR_PATH_PIPELINE         the same pipeline with 16 KiB tiles (highest
 *                            bandwidth on large messages).
 * By default the path comes from tables measured on GB300 per call shape --
 * dtype, stage mode (encode-only, one-stage, two-stage), W and format -- as
 * two size limits: messages of at most the direct limit (elements per rank)
 * take the direct kernel, those of at most the narrow-tile limit the
 * narrow-tile pipeline, longer ones the wide-tile pipeline.  This is the
 * counterpart, for this data path, of the per-(dtype, world size) size
 * thresholds _QR_MIN_SIZE on the vLLM quick_all_reduce page and of the size
 * rule in vLLM PR #18473's description (the tables: csrc/qr_select_table.h,
 * generated by select_table.py from the committed sweep).  The narrow-tile
 * pipeline is built for W <= 4; a W = 8 call sent there runs wide tiles.
 *
 * qr_kernel_path returns the path a call of the given shape and size takes
 * now (stages 0: qr_quantize, W ignored; 1 or 2: the allreduce), or -1 for a
 * shape no call can have.  qr_set_kernel_path(path) forces one path for
 * EVERY call in the whole process until qr_set_kernel_path(QR_PATH_TABLE)
 * restores the tables (QR_ERR_PATH for any other value; the setting is then
 * unchanged).  It is process-global state: a caller in another thread is
 * rerouted too (results stay bit-identical; only timing changes).
 * qr_forced_kernel_path returns the forced path, or QR_PATH_TABLE.  Host
 * only, no CUDA call; thread-safe (one atomic word). */
typedef enum {
  QR_PATH_TABLE = -1,
  QR_PATH_DIRECT = 0,
  QR_PATH_PIPELINE_NARROW = 1,
  QR_PATH_PIPELINE = 2
} qr_path;
int qr_kernel_path(int W, qr_dtype dt, qr_format fmt, int stages, size_t n);
qr_status qr_set_kernel_path(int path);
int qr_forced_kernel_path(void);

/* A short English description of a status code (static storage). */
const char *qr_status_string(qr_status st);

/* Self-test of the kernels' bounded waits, for tests of the failure path:
 * launches one warp that waits on a shared-memory barrier nothing will
 * complete, through the same bounded-wait routine the pipeline kernel uses,
 * with a limit of limit_us microseconds (1 .. 1000000; otherwise
 * QR_ERR_SIZE).  When the limit expires the wait gives up, the kernel sets
 * flag 8 in the device flag word and returns; read it with
 * qr_device_error().  Nothing faults and nothing hangs. */
qr_status qr_selftest_wait_timeout(unsigned int limit_us, void *stream);

/* Self-test of the block-scale reciprocal the direct path's allreduce
 * kernels and the pipeline kernel at W = 2 and 4 use (two
 * Newton-Raphson steps on the hardware approximation instead of the
 * correctly rounded library reciprocal): writes, for every positive finite
 * fp16 value s (bit patterns 1 .. 0x7BFF in order), the binary32 reciprocal
 * the kernels would use for a block scale s, so that a test can compare all
 * of them with the IEEE quotient 1/s that the method defines.
 *   out     device, QR_SELFTEST_RECIPROCALS floats, 16-byte aligned, written
 * QR_ERR_NULL / QR_ERR_ALIGN for a bad buffer; asynchronous on `stream`. */
#define QR_SELFTEST_RECIPROCALS 0x7BFF
qr_status qr_selftest_reciprocal(float *out, void *stream);

/* Kernels never wait forever: a pipeline wait that exceeds its time limit
 * sets a flag in device memory and the kernel returns early.  This call
 * synchronises the current device, copies the flags to *flags (0 = none
 * raised; 1 = a consumer wait, 2 = a producer wait, 4 = the final drain,
 * 8 = the self-test) and clears them when clear != 0.  Returns QR_ERR_DEVICE when a
 * flag was raised, QR_OK otherwise, QR_ERR_CUDA on a CUDA error. */
qr_status qr_device_error(unsigned int *flags, int clear);

#ifdef __cplusplus
}
#endif
#endif /* QR_H */
