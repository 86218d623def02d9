// qr_api.cu -- the C ABI of libqr.so (declared in include/qr.h): argument
// validation, encoded-buffer layout, dispatch to the per-format launchers.
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "qr.h"
#include "qr_launch.h"
#include "qr_select_table.h"

namespace qr {

__device__ unsigned g_qr_error_flags;

namespace {

constexpr int kMaxDevices = 64;

int code_bits(int fmt) {
  switch (fmt) {
    case FMT_Q8: case FMT_FP8: case FMT_Q8A: return 8;
    case FMT_Q6: return 6;
    case FMT_Q4: case FMT_Q4A: return 4;
    default: return 0;
  }
}
bool is_asym(int fmt) { return fmt == FMT_Q8A || fmt == FMT_Q4A; }
bool valid_format(int fmt) { return fmt >= FMT_FP && fmt <= FMT_Q4A; }
bool valid_dtype(int dt) { return dt == DT_F16 || dt == DT_BF16; }
bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool overlap(const void* a, size_t na, const void* b, size_t nb) {
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return na && nb && x < y + nb && y < x + na;
}

qr_status check_size(size_t n) {
  if (n > QR_MAX_ELEMS) return QR_ERR_SIZE;
  if ((n * 2) % 16 != 0) return QR_ERR_SIZE;  // byte size a multiple of 16
  return QR_OK;
}

qr_status to_status(cudaError_t e) { return e == cudaSuccess ? QR_OK : QR_ERR_CUDA; }

// Kernel-path selection: the measured tables, or a process-wide forced path
// (QR_PATH_TABLE: none).
std::atomic<int> g_forced_path{QR_PATH_TABLE};

int world_index(int W) { return W == 1 ? 0 : W == 2 ? 1 : W == 4 ? 2 : 3; }

// The kernel a call of this shape and size runs: the direct kernel up to the
// direct limit, the narrow-tile pipeline up to the narrow-tile limit, the
// wide-tile pipeline beyond.
int select_path(int dt, int mode, int W, int fmt, unsigned long long n) {
  const int forced = g_forced_path.load(std::memory_order_relaxed);
  if (forced != QR_PATH_TABLE) return forced;
  const int w = world_index(W);
  if (n <= kDirectLimitTable[dt][mode][w][fmt]) return QR_PATH_DIRECT;
  if (n <= kNarrowTileLimitTable[dt][mode][w][fmt]) return QR_PATH_PIPELINE_NARROW;
  return QR_PATH_PIPELINE;
}

cudaError_t dispatch_direct(int fmt, int dt, int mode, const PipeParams& p, cudaStream_t s) {
  switch (fmt) {
    case 0: return launch_direct_fmt_0(dt, mode, p, s);
    case 1: return launch_direct_fmt_1(dt, mode, p, s);
    case 2: return launch_direct_fmt_2(dt, mode, p, s);
    case 3: return launch_direct_fmt_3(dt, mode, p, s);
    case 4: return launch_direct_fmt_4(dt, mode, p, s);
    case 5: return launch_direct_fmt_5(dt, mode, p, s);
    case 6: return launch_direct_fmt_6(dt, mode, p, s);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t dispatch_pipeline(int fmt, int dt, int mode, const PipeParams& p, cudaStream_t s) {
  const int path = select_path(dt, mode, p.W, fmt, p.n);
  if (path == QR_PATH_DIRECT) return dispatch_direct(fmt, dt, mode, p, s);
  const int cw = path == QR_PATH_PIPELINE_NARROW ? kNarrowTile : kWideTile;
  switch (fmt) {
    case 0: return launch_pipeline_fmt_0(dt, mode, cw, p, s);
    case 1: return launch_pipeline_fmt_1(dt, mode, cw, p, s);
    case 2: return launch_pipeline_fmt_2(dt, mode, cw, p, s);
    case 3: return launch_pipeline_fmt_3(dt, mode, cw, p, s);
    case 4: return launch_pipeline_fmt_4(dt, mode, cw, p, s);
    case 5: return launch_pipeline_fmt_5(dt, mode, cw, p, s);
    case 6: return launch_pipeline_fmt_6(dt, mode, cw, p, s);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t dispatch_decode(int fmt, int dt, const DecodeParams& p, cudaStream_t s) {
  switch (fmt) {
    case 0: return launch_decode_fmt_0(dt, p, s);
    case 1: return launch_decode_fmt_1(dt, p, s);
    case 2: return launch_decode_fmt_2(dt, p, s);
    case 3: return launch_decode_fmt_3(dt, p, s);
    case 4: return launch_decode_fmt_4(dt, p, s);
    case 5: return launch_decode_fmt_5(dt, p, s);
    case 6: return launch_decode_fmt_6(dt, p, s);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t dispatch_staged(int fmt, int dt, const StagedParams& p, const DecodeParams& dp, cudaStream_t s) {
  switch (fmt) {
    case 0: return launch_staged_fmt_0(dt, p, dp, s);
    case 1: return launch_staged_fmt_1(dt, p, dp, s);
    case 2: return launch_staged_fmt_2(dt, p, dp, s);
    case 3: return launch_staged_fmt_3(dt, p, dp, s);
    case 4: return launch_staged_fmt_4(dt, p, dp, s);
    case 5: return launch_staged_fmt_5(dt, p, dp, s);
    case 6: return launch_staged_fmt_6(dt, p, dp, s);
    default: return cudaErrorInvalidValue;
  }
}

// Stage-1 slot geometry: chunk_nb = ceil(nb / W) blocks per owner; a slot is
// one encoded sub-message of chunk_nb blocks, padded to 16 bytes.
void staged_geometry(int W, int fmt, size_t n, size_t* chunk_nb, size_t* slot_bytes) {
  const size_t nb = (n + 31) / 32;
  *chunk_nb = (nb + W - 1) / W;
  size_t per_block = fmt == FMT_FP ? 64 : 32 * static_cast<size_t>(code_bits(fmt)) / 8 + 2 + (is_asym(fmt) ? 2 : 0);
  *slot_bytes = (*chunk_nb * per_block + 15) / 16 * 16;
}

// Encoded layout: codes[nb][cb] | scales[nb] | zps[nb] (asymmetric only).
void encoded_regions(int fmt, size_t n, void* base, uint8_t** codes, uint16_t** scales, uint16_t** zps,
                     uint16_t** fp_values) {
  *codes = nullptr;
  *scales = *zps = *fp_values = nullptr;
  if (!base) return;
  if (fmt == FMT_FP) {
    *fp_values = static_cast<uint16_t*>(base);
    return;
  }
  const size_t nb = (n + 31) / 32;
  const size_t cb = 32 * static_cast<size_t>(code_bits(fmt)) / 8;
  uint8_t* b = static_cast<uint8_t*>(base);
  *codes = b;
  *scales = reinterpret_cast<uint16_t*>(b + nb * cb);
  if (is_asym(fmt)) *zps = reinterpret_cast<uint16_t*>(b + nb * cb + 2 * nb);
}

// One warp waits on a shared-memory barrier that nothing will complete; the
// bounded wait gives up after limit_ns and raises kErrSelfTest.
__global__ void qr_selftest_wait_kernel(unsigned* err, unsigned long long limit_ns) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  const bool completed = mbar_wait(&bar, 0u, limit_ns);
  if (!__all_sync(0xffffffffu, completed) && threadIdx.x == 0) atomicOr(err, kErrSelfTest);
}

// The block-scale reciprocal of every positive finite fp16 value (bit
// patterns 1 .. 0x7BFF, in order) into out.
__global__ void qr_selftest_reciprocal_kernel(float* out) {
  const unsigned i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < QR_SELFTEST_RECIPROCALS)
    out[i] = recip_of_half(__half2float(__ushort_as_half(static_cast<unsigned short>(i + 1))));
}

// ---- qr_allreduce_host: per-device copy streams and reusable events ----
// Chunk i uses buffer i & 1.  in_done[b]: its copy-in finished; k_done[b]:
// its kernel finished (the inputs may be overwritten); out_done[b]: its
// copy-out finished (the output may be overwritten).
struct HostPipe {
  bool ready = false;
  cudaStream_t s_in = nullptr, s_out = nullptr;
  cudaEvent_t start = nullptr;
  cudaEvent_t in_done[2] = {nullptr, nullptr}, k_done[2] = {nullptr, nullptr}, out_done[2] = {nullptr, nullptr};
};
HostPipe g_host_pipe[kMaxDevices];
std::mutex g_host_mutex[kMaxDevices];

cudaError_t host_pipe_ready(HostPipe& h) {
  if (h.ready) return cudaSuccess;
  cudaError_t e = cudaStreamCreateWithFlags(&h.s_in, cudaStreamNonBlocking);
  if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&h.s_out, cudaStreamNonBlocking);
  if (e == cudaSuccess) e = cudaEventCreateWithFlags(&h.start, cudaEventDisableTiming);
  for (int b = 0; b < 2 && e == cudaSuccess; ++b) {
    e = cudaEventCreateWithFlags(&h.in_done[b], cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&h.k_done[b], cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&h.out_done[b], cudaEventDisableTiming);
  }
  if (e != cudaSuccess) {  // release what was made; the next call tries again
    if (h.s_in) cudaStreamDestroy(h.s_in);
    if (h.s_out) cudaStreamDestroy(h.s_out);
    cudaEvent_t* evs[] = {&h.start, &h.in_done[0], &h.in_done[1], &h.k_done[0], &h.k_done[1], &h.out_done[0],
                          &h.out_done[1]};
    for (cudaEvent_t* ev : evs)
      if (*ev) cudaEventDestroy(*ev);
    h = HostPipe();
    return e;
  }
  h.ready = true;
  return cudaSuccess;
}

size_t pad256(size_t bytes) { return (bytes + 255) / 256 * 256; }

// One chunk buffer of the host-entry workspace: W inputs | output | payload.
size_t host_chunk_buffer_bytes(int W, int fmt, size_t chunk) {
  return static_cast<size_t>(W + 1) * pad256(chunk * 2) + pad256(qr_encoded_bytes(static_cast<qr_format>(fmt), chunk));
}

}  // namespace

unsigned* device_error_word() {
  // one atomic pointer per device: racing first calls each look the address
  // up and publish the same value
  static std::atomic<unsigned*> addr[kMaxDevices];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  unsigned* a = addr[dev].load(std::memory_order_acquire);
  if (!a) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_qr_error_flags) != cudaSuccess || !p) return nullptr;
    a = static_cast<unsigned*>(p);
    addr[dev].store(a, std::memory_order_release);
  }
  return a;
}

qr_status staged_check_args(int W, int dt, int fmt, size_t n) {
  if (!valid_dtype(dt)) return QR_ERR_DTYPE;
  if (!valid_format(fmt)) return QR_ERR_FORMAT;
  if (W != 1 && W != 2 && W != 4 && W != 8) return QR_ERR_WORLD;
  return check_size(n);
}

qr_status staged_check_buffers(int W, int fmt, const void* const* inputs, size_t n, const void* out,
                               const void* wire, const void* stage1) {
  for (int r = 0; r < W; ++r)
    if (!inputs[r]) return QR_ERR_NULL;
  if (!aligned16(out) || !aligned16(wire) || (stage1 && !aligned16(stage1))) return QR_ERR_ALIGN;
  for (int r = 0; r < W; ++r)
    if (!aligned16(inputs[r])) return QR_ERR_ALIGN;
  const qr_format fm = static_cast<qr_format>(fmt);
  const size_t msg = n * 2, wbytes = qr_encoded_bytes(fm, n), sbytes = stage1 ? qr_stage1_bytes(W, fm, n) : 0;
  for (int r = 0; r < W; ++r)
    if (overlap(inputs[r], msg, out, msg) || overlap(inputs[r], msg, wire, wbytes) ||
        overlap(inputs[r], msg, stage1, sbytes))
      return QR_ERR_OVERLAP;
  if (overlap(out, msg, wire, wbytes) || overlap(out, msg, stage1, sbytes) || overlap(wire, wbytes, stage1, sbytes))
    return QR_ERR_OVERLAP;
  return QR_OK;
}

qr_status staged_launch(int W, int dt, int fmt, const void* const* inputs, size_t n, void* out, void* wire,
                        uint8_t* stage1, cudaStream_t s) {
  StagedParams p;
  std::memset(&p, 0, sizeof p);
  p.one = 1.0f;
  for (int r = 0; r < W; ++r) p.in[r] = inputs[r];
  p.W = W;
  p.n = n;
  p.nb = (n + 31) / 32;
  size_t chunk_nb, slot_bytes;
  staged_geometry(W, fmt, n, &chunk_nb, &slot_bytes);
  p.chunk_nb = chunk_nb;
  p.slot_bytes = slot_bytes;
  p.stage1 = stage1;
  encoded_regions(fmt, n, wire, &p.codes, &p.scales, &p.zps, &p.fp_values);

  DecodeParams dp;
  std::memset(&dp, 0, sizeof dp);
  dp.codes = p.codes;
  dp.scales = p.scales;
  dp.zps = p.zps;
  dp.fp_values = p.fp_values;
  dp.out = out;
  dp.n = n;
  dp.nb = p.nb;
  dp.err = device_error_word();
  if (!dp.err) return QR_ERR_CUDA;
  return to_status(dispatch_staged(fmt, dt, p, dp, s));
}

}  // namespace qr

using namespace qr;

extern "C" {

size_t qr_encoded_bytes(qr_format fmt, size_t n) {
  const int f = static_cast<int>(fmt);
  if (!valid_format(f)) return 0;
  if (f == FMT_FP) return n * 2;
  const size_t nb = (n + 31) / 32;
  return nb * (32 * static_cast<size_t>(code_bits(f)) / 8 + 2 + (is_asym(f) ? 2 : 0));
}

const char* qr_status_string(qr_status st) {
  switch (st) {
    case QR_OK: return "ok";
    case QR_ERR_NULL: return "a required pointer is NULL";
    case QR_ERR_DTYPE: return "dtype must be fp16 or bf16";
    case QR_ERR_FORMAT: return "unknown format";
    case QR_ERR_WORLD: return "world size must be 1, 2, 4 or 8";
    case QR_ERR_STAGES: return "stages must be 1 or 2 (and wire must be NULL for 1)";
    case QR_ERR_SIZE: return "message byte size must be a multiple of 16 (and n <= 2^36)";
    case QR_ERR_ALIGN: return "buffers must be 16-byte aligned";
    case QR_ERR_OVERLAP: return "an output buffer overlaps an input or another output";
    case QR_ERR_CUDA: return "CUDA runtime error";
    case QR_ERR_DEVICE: return "a kernel gave up waiting on its pipeline";
    case QR_ERR_SCRATCH: return "the message needs more stage-1 space than the built-in scratch array holds";
    case QR_ERR_PATH: return "not a kernel path (QR_PATH_TABLE, QR_PATH_DIRECT, QR_PATH_PIPELINE_NARROW, QR_PATH_PIPELINE)";
    default: return "unknown status";
  }
}

qr_status qr_quantize(qr_dtype dt, qr_format fmt, const void* in, size_t n, void* enc, void* stream) {
  const int f = static_cast<int>(fmt), d = static_cast<int>(dt);
  if (n && (!in || !enc)) return QR_ERR_NULL;
  if (!valid_dtype(d)) return QR_ERR_DTYPE;
  if (!valid_format(f)) return QR_ERR_FORMAT;
  qr_status st = check_size(n);
  if (st != QR_OK) return st;
  if (n == 0) return QR_OK;
  if (!aligned16(in) || !aligned16(enc)) return QR_ERR_ALIGN;
  if (overlap(in, n * 2, enc, qr_encoded_bytes(fmt, n))) return QR_ERR_OVERLAP;

  PipeParams p;
  std::memset(&p, 0, sizeof p);
  p.one = 1.0f;
  p.in[0] = in;
  p.W = 1;
  p.n = n;
  p.nb = (n + 31) / 32;
  encoded_regions(f, n, enc, &p.codes, &p.scales, &p.zps, &p.fp_values);
  p.err = device_error_word();
  if (!p.err) return QR_ERR_CUDA;
  return to_status(dispatch_pipeline(f, d, MODE_ENCODE, p, static_cast<cudaStream_t>(stream)));
}

qr_status qr_dequantize(qr_dtype dt, qr_format fmt, const void* enc, size_t n, void* out, void* stream) {
  const int f = static_cast<int>(fmt), d = static_cast<int>(dt);
  if (n && (!enc || !out)) return QR_ERR_NULL;
  if (!valid_dtype(d)) return QR_ERR_DTYPE;
  if (!valid_format(f)) return QR_ERR_FORMAT;
  qr_status st = check_size(n);
  if (st != QR_OK) return st;
  if (n == 0) return QR_OK;
  if (!aligned16(enc) || !aligned16(out)) return QR_ERR_ALIGN;
  if (overlap(enc, qr_encoded_bytes(fmt, n), out, n * 2)) return QR_ERR_OVERLAP;

  DecodeParams p;
  std::memset(&p, 0, sizeof p);
  uint8_t* codes;
  uint16_t *scales, *zps, *fpv;
  encoded_regions(f, n, const_cast<void*>(enc), &codes, &scales, &zps, &fpv);
  p.codes = codes;
  p.scales = scales;
  p.zps = zps;
  p.fp_values = fpv;
  p.out = out;
  p.n = n;
  p.nb = (n + 31) / 32;
  p.err = device_error_word();
  if (!p.err) return QR_ERR_CUDA;
  return to_status(dispatch_decode(f, d, p, static_cast<cudaStream_t>(stream)));
}

qr_status qr_allreduce_emulated(int W, qr_dtype dt, qr_format fmt, int stages, const void* const* inputs,
                                size_t n, void* out, void* wire, void* stream) {
  const int f = static_cast<int>(fmt), d = static_cast<int>(dt);
  if (n && (!inputs || !out)) return QR_ERR_NULL;
  if (!valid_dtype(d) && d != DT_BF16_AS_F16) return QR_ERR_DTYPE;
  if (!valid_format(f)) return QR_ERR_FORMAT;
  if (W != 1 && W != 2 && W != 4 && W != 8) return QR_ERR_WORLD;
  if (stages != 1 && stages != 2) return QR_ERR_STAGES;
  if (stages == 1 && wire) return QR_ERR_STAGES;
  qr_status st = check_size(n);
  if (st != QR_OK) return st;
  if (n == 0) return QR_OK;
  for (int r = 0; r < W; ++r)
    if (!inputs[r]) return QR_ERR_NULL;
  if (!aligned16(out) || (wire && !aligned16(wire))) return QR_ERR_ALIGN;
  for (int r = 0; r < W; ++r)
    if (!aligned16(inputs[r])) return QR_ERR_ALIGN;
  const size_t msg = n * 2, wbytes = wire ? qr_encoded_bytes(fmt, n) : 0;
  for (int r = 0; r < W; ++r)
    if (overlap(inputs[r], msg, out, msg) || overlap(inputs[r], msg, wire, wbytes)) return QR_ERR_OVERLAP;
  if (overlap(out, msg, wire, wbytes)) return QR_ERR_OVERLAP;

  PipeParams p;
  std::memset(&p, 0, sizeof p);
  p.one = 1.0f;
  for (int r = 0; r < W; ++r) p.in[r] = inputs[r];
  p.W = W;
  p.n = n;
  p.nb = (n + 31) / 32;
  p.out = out;
  if (stages == 2) encoded_regions(f, n, wire, &p.codes, &p.scales, &p.zps, &p.fp_values);
  p.err = device_error_word();
  if (!p.err) return QR_ERR_CUDA;
  const int mode = stages == 1 ? MODE_AR1 : MODE_AR2;
  return to_status(dispatch_pipeline(f, d, mode, p, static_cast<cudaStream_t>(stream)));
}

size_t qr_stage1_bytes(int W, qr_format fmt, size_t n) {
  const int f = static_cast<int>(fmt);
  if ((W != 1 && W != 2 && W != 4 && W != 8) || !valid_format(f)) return 0;
  size_t chunk_nb, slot_bytes;
  staged_geometry(W, f, n, &chunk_nb, &slot_bytes);
  return static_cast<size_t>(W) * W * slot_bytes;
}

qr_status qr_allreduce_staged(int W, qr_dtype dt, qr_format fmt, const void* const* inputs, size_t n, void* out,
                              void* wire, void* stage1, void* stream) {
  const int f = static_cast<int>(fmt), d = static_cast<int>(dt);
  if (n && (!inputs || !out || !wire || !stage1)) return QR_ERR_NULL;
  qr_status st = staged_check_args(W, d, f, n);
  if (st != QR_OK) return st;
  if (n == 0) return QR_OK;
  st = staged_check_buffers(W, f, inputs, n, out, wire, stage1);
  if (st != QR_OK) return st;
  return staged_launch(W, d, f, inputs, n, out, wire, static_cast<uint8_t*>(stage1),
                       static_cast<cudaStream_t>(stream));
}

size_t qr_host_workspace_bytes(int W, qr_format fmt, size_t chunk_elems) {
  const int f = static_cast<int>(fmt);
  if ((W != 1 && W != 2 && W != 4 && W != 8) || !valid_format(f)) return 0;
  if (chunk_elems == 0 || chunk_elems % 32 != 0 || chunk_elems > QR_MAX_ELEMS) return 0;
  return 2 * host_chunk_buffer_bytes(W, f, chunk_elems);
}

qr_status qr_allreduce_host(int W, qr_dtype dt, qr_format fmt, int stages, const void* const* host_inputs,
                            size_t n, void* host_out, void* host_wire, void* workspace, size_t workspace_bytes,
                            size_t chunk_elems, void* stream) {
  const int f = static_cast<int>(fmt), d = static_cast<int>(dt);
  if (n && (!host_inputs || !host_out || !workspace)) return QR_ERR_NULL;
  if (!valid_dtype(d) && d != DT_BF16_AS_F16) return QR_ERR_DTYPE;
  if (!valid_format(f)) return QR_ERR_FORMAT;
  if (W != 1 && W != 2 && W != 4 && W != 8) return QR_ERR_WORLD;
  if (stages != 1 && stages != 2) return QR_ERR_STAGES;
  if (stages == 1 && host_wire) return QR_ERR_STAGES;
  qr_status st = check_size(n);
  if (st != QR_OK) return st;
  const size_t need = qr_host_workspace_bytes(W, fmt, chunk_elems);
  if (need == 0 || workspace_bytes < need) return QR_ERR_SIZE;
  if (n == 0) return QR_OK;
  for (int r = 0; r < W; ++r)
    if (!host_inputs[r]) return QR_ERR_NULL;
  if (!aligned16(workspace)) return QR_ERR_ALIGN;
  const size_t msg = n * 2, wbytes = host_wire ? qr_encoded_bytes(fmt, n) : 0;
  for (int r = 0; r < W; ++r)
    if (overlap(host_inputs[r], msg, host_out, msg) || overlap(host_inputs[r], msg, host_wire, wbytes))
      return QR_ERR_OVERLAP;
  if (overlap(host_out, msg, host_wire, wbytes)) return QR_ERR_OVERLAP;

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return QR_ERR_CUDA;
  unsigned* err = device_error_word();
  if (!err) return QR_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_host_mutex[dev]);
  HostPipe& h = g_host_pipe[dev];
  if (host_pipe_ready(h) != cudaSuccess) return QR_ERR_CUDA;

  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  const size_t nb = (n + 31) / 32;
  const size_t cb = 32 * static_cast<size_t>(code_bits(f)) / 8;
  const size_t buf_bytes = host_chunk_buffer_bytes(W, f, chunk_elems);
  const size_t nchunks = (n + chunk_elems - 1) / chunk_elems;
  const int mode = stages == 1 ? MODE_AR1 : MODE_AR2;
  uint8_t* hwire = static_cast<uint8_t*>(host_wire);
  uint8_t* hout = static_cast<uint8_t*>(host_out);

#define QR_TRY(call)                               \
  do {                                             \
    if ((call) != cudaSuccess) return QR_ERR_CUDA; \
  } while (0)
  // both copy streams start after the work already on `stream`
  QR_TRY(cudaEventRecord(h.start, s));
  QR_TRY(cudaStreamWaitEvent(h.s_in, h.start, 0));
  QR_TRY(cudaStreamWaitEvent(h.s_out, h.start, 0));
  for (size_t i = 0; i < nchunks; ++i) {
    const int b = static_cast<int>(i & 1);
    uint8_t* base = static_cast<uint8_t*>(workspace) + b * buf_bytes;
    uint8_t* d_out = base + static_cast<size_t>(W) * pad256(chunk_elems * 2);
    uint8_t* d_wire = d_out + pad256(chunk_elems * 2);
    const size_t c0 = i * chunk_elems;
    const size_t cn = (n - c0) < chunk_elems ? (n - c0) : chunk_elems;
    const size_t blk0 = c0 / 32, nbc = (cn + 31) / 32;

    // copy-in: buffer b is free once chunk i-2's kernel has read it
    if (i >= 2) QR_TRY(cudaStreamWaitEvent(h.s_in, h.k_done[b], 0));
    for (int r = 0; r < W; ++r)
      QR_TRY(cudaMemcpyAsync(base + r * pad256(chunk_elems * 2), static_cast<const uint8_t*>(host_inputs[r]) + c0 * 2,
                             cn * 2, cudaMemcpyHostToDevice, h.s_in));
    QR_TRY(cudaEventRecord(h.in_done[b], h.s_in));

    // kernel on the caller's stream: after the copy-in, and after chunk i-2's
    // copy-out has read this buffer's output and payload
    QR_TRY(cudaStreamWaitEvent(s, h.in_done[b], 0));
    if (i >= 2) QR_TRY(cudaStreamWaitEvent(s, h.out_done[b], 0));
    PipeParams p;
    std::memset(&p, 0, sizeof p);
    p.one = 1.0f;
    for (int r = 0; r < W; ++r) p.in[r] = base + r * pad256(chunk_elems * 2);
    p.W = W;
    p.n = cn;
    p.nb = nbc;
    p.out = d_out;
    if (stages == 2 && host_wire) encoded_regions(f, cn, d_wire, &p.codes, &p.scales, &p.zps, &p.fp_values);
    p.err = err;
    QR_TRY(dispatch_pipeline(f, d, mode, p, s));
    QR_TRY(cudaEventRecord(h.k_done[b], s));

    // copy-out into the message-wide host layout
    QR_TRY(cudaStreamWaitEvent(h.s_out, h.k_done[b], 0));
    QR_TRY(cudaMemcpyAsync(hout + c0 * 2, d_out, cn * 2, cudaMemcpyDeviceToHost, h.s_out));
    if (hwire) {
      if (f == FMT_FP) {
        QR_TRY(cudaMemcpyAsync(hwire + c0 * 2, d_wire, cn * 2, cudaMemcpyDeviceToHost, h.s_out));
      } else {
        QR_TRY(cudaMemcpyAsync(hwire + blk0 * cb, d_wire, nbc * cb, cudaMemcpyDeviceToHost, h.s_out));
        QR_TRY(cudaMemcpyAsync(hwire + nb * cb + blk0 * 2, d_wire + nbc * cb, nbc * 2, cudaMemcpyDeviceToHost,
                               h.s_out));
        if (is_asym(f))
          QR_TRY(cudaMemcpyAsync(hwire + nb * cb + nb * 2 + blk0 * 2, d_wire + nbc * cb + nbc * 2, nbc * 2,
                                 cudaMemcpyDeviceToHost, h.s_out));
      }
    }
    QR_TRY(cudaEventRecord(h.out_done[b], h.s_out));
  }
  // the caller's stream continues after the last copy-out (the copy-out
  // stream runs in order, so that covers every chunk)
  QR_TRY(cudaStreamWaitEvent(s, h.out_done[(nchunks - 1) & 1], 0));
#undef QR_TRY
  return QR_OK;
}

int qr_kernel_path(int W, qr_dtype dt, qr_format fmt, int stages, size_t n) {
  const int d = static_cast<int>(dt), f = static_cast<int>(fmt);
  if (!valid_format(f) || stages < 0 || stages > 2) return -1;
  if (stages == 0) {  // qr_quantize: one rank, fp16 or bf16
    if (!valid_dtype(d)) return -1;
    return select_path(d, MODE_ENCODE, 1, f, n);
  }
  if (!valid_dtype(d) && d != DT_BF16_AS_F16) return -1;
  if (W != 1 && W != 2 && W != 4 && W != 8) return -1;
  return select_path(d, stages == 1 ? MODE_AR1 : MODE_AR2, W, f, n);
}

qr_status qr_set_kernel_path(int path) {
  if (path != QR_PATH_TABLE && path != QR_PATH_DIRECT && path != QR_PATH_PIPELINE_NARROW && path != QR_PATH_PIPELINE)
    return QR_ERR_PATH;
  g_forced_path.store(path);
  return QR_OK;
}

int qr_forced_kernel_path(void) { return g_forced_path.load(); }

qr_status qr_selftest_wait_timeout(unsigned int limit_us, void* stream) {
  if (limit_us == 0 || limit_us > 1000000u) return QR_ERR_SIZE;
  unsigned* err = device_error_word();
  if (!err) return QR_ERR_CUDA;
  qr_selftest_wait_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(
      err, static_cast<unsigned long long>(limit_us) * 1000ull);
  return to_status(cudaGetLastError());
}

qr_status qr_selftest_reciprocal(float* out, void* stream) {
  if (!out) return QR_ERR_NULL;
  if (!aligned16(out)) return QR_ERR_ALIGN;
  qr_selftest_reciprocal_kernel<<<(QR_SELFTEST_RECIPROCALS + 255) / 256, 256, 0, static_cast<cudaStream_t>(stream)>>>(out);
  return to_status(cudaGetLastError());
}

qr_status qr_device_error(unsigned int* flags, int clear) {
  if (cudaDeviceSynchronize() != cudaSuccess) return QR_ERR_CUDA;
  unsigned v = 0;
  if (cudaMemcpyFromSymbol(&v, g_qr_error_flags, sizeof v) != cudaSuccess) return QR_ERR_CUDA;
  if (clear) {
    const unsigned zero = 0;
    if (cudaMemcpyToSymbol(g_qr_error_flags, &zero, sizeof zero) != cudaSuccess) return QR_ERR_CUDA;
  }
  if (flags) *flags = v;
  return v ? QR_ERR_DEVICE : QR_OK;
}

}  // extern "C"
