// qr_noalloc.cu -- qr_allreduce_staged_noalloc: the staged two-stage
// allreduce for callers that cannot allocate device memory.
//
// qr_allreduce_staged needs a stage-1 exchange buffer from its caller.  Some
// callers cannot get one: code that runs while a CUDA graph is being
// captured (an allocation is not an operation a stream can record), a plugin
// or callback that is handed only its input and output pointers and must not
// go around its host framework's memory allocator, or a latency-critical path
// where cudaMalloc/cudaFree (and the device synchronisation cudaFree implies)
// are not allowed.  This entry point takes no scratch argument: the stage-1
// buffer is a fixed array in device memory that is part of this library, so
// nothing is allocated per call.
//
// The array is a file-scope __device__ variable: every GPU on which the
// library is used holds its kNoAllocScratchBytes until the process exits.
// Host code cannot use the array's name as a device address (on the host it
// names a stand-in object), so the first call on each device looks the
// address up with cudaGetSymbolAddress, with that device current, and keeps
// it for later calls.
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>
#include <cstring>

#include "qr.h"
#include "qr_launch.h"

namespace qr {
namespace {

constexpr size_t kNoAllocScratchBytes = QR_NOALLOC_SCRATCH_BYTES;
constexpr int kMaxNoAllocDevices = 64;

static __device__ __align__(256) uint8_t g_qr_noalloc_scratch[kNoAllocScratchBytes];

std::atomic<uint8_t*> g_scratch_addr[kMaxNoAllocDevices];

// Device address of the scratch array on the current device (looked up once
// per device); nullptr on a CUDA error.
uint8_t* scratch_address() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxNoAllocDevices) return nullptr;
  uint8_t* p = g_scratch_addr[dev].load(std::memory_order_acquire);
  if (p) return p;
  void* addr = nullptr;
  if (cudaGetSymbolAddress(&addr, g_qr_noalloc_scratch) != cudaSuccess || !addr) return nullptr;
  p = static_cast<uint8_t*>(addr);
  g_scratch_addr[dev].store(p, std::memory_order_release);
  return p;
}

bool is_asym_fmt(int f) { return f == FMT_Q8A || f == FMT_Q4A; }

cudaError_t launch_staged(int fmt, int dt, const StagedParams& p, const DecodeParams& dp, cudaStream_t s) {
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

bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return na && nb && x < y + nb && y < x + na;
}

}  // namespace
}  // namespace qr

using namespace qr;

extern "C" qr_status qr_allreduce_staged_noalloc(int W, qr_dtype dt, qr_format fmt, const void* const* inputs,
                                                 size_t n, void* out, void* wire, void* stream) {
  const int f = static_cast<int>(fmt), d = static_cast<int>(dt);
  if (n && (!inputs || !out || !wire)) return QR_ERR_NULL;
  if (d != DT_F16 && d != DT_BF16) return QR_ERR_DTYPE;
  if (f < FMT_FP || f > FMT_Q4A) return QR_ERR_FORMAT;
  if (W != 1 && W != 2 && W != 4 && W != 8) return QR_ERR_WORLD;
  if (n > QR_MAX_ELEMS || (n * 2) % 16 != 0) return QR_ERR_SIZE;
  if (n == 0) return QR_OK;
  const size_t need = qr_stage1_bytes(W, fmt, n);
  if (need > kNoAllocScratchBytes) return QR_ERR_SCRATCH;
  for (int r = 0; r < W; ++r)
    if (!inputs[r]) return QR_ERR_NULL;
  auto aligned = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
  if (!aligned(out) || !aligned(wire)) return QR_ERR_ALIGN;
  for (int r = 0; r < W; ++r)
    if (!aligned(inputs[r])) return QR_ERR_ALIGN;
  const size_t msg = n * 2, wbytes = qr_encoded_bytes(fmt, n);
  for (int r = 0; r < W; ++r)
    if (overlaps(inputs[r], msg, out, msg) || overlaps(inputs[r], msg, wire, wbytes)) return QR_ERR_OVERLAP;
  if (overlaps(out, msg, wire, wbytes)) return QR_ERR_OVERLAP;

  uint8_t* scratch = scratch_address();
  if (!scratch) return QR_ERR_CUDA;
  // Same geometry and regions as qr_allreduce_staged (see qr_stage1_bytes).
  const size_t nb = (n + 31) / 32;
  const size_t chunk_nb = (nb + W - 1) / W;
  const size_t per_block =
      f == FMT_FP ? 64 : 32 * static_cast<size_t>(f == FMT_Q6 ? 6 : (f == FMT_Q4 || f == FMT_Q4A) ? 4 : 8) / 8 + 2 +
                             (is_asym_fmt(f) ? 2 : 0);
  StagedParams p;
  std::memset(&p, 0, sizeof p);
  p.one = 1.0f;
  for (int r = 0; r < W; ++r) p.in[r] = inputs[r];
  p.W = W;
  p.n = n;
  p.nb = nb;
  p.chunk_nb = chunk_nb;
  p.slot_bytes = (chunk_nb * per_block + 15) / 16 * 16;
  p.stage1 = scratch;
  uint8_t* wb = static_cast<uint8_t*>(wire);
  if (f == FMT_FP) {
    p.fp_values = static_cast<uint16_t*>(wire);
  } else {
    const size_t cb = per_block - 2 - (is_asym_fmt(f) ? 2 : 0);
    p.codes = wb;
    p.scales = reinterpret_cast<uint16_t*>(wb + nb * cb);
    if (is_asym_fmt(f)) p.zps = reinterpret_cast<uint16_t*>(wb + nb * cb + 2 * nb);
  }
  DecodeParams dp;
  std::memset(&dp, 0, sizeof dp);
  dp.codes = p.codes;
  dp.scales = p.scales;
  dp.zps = p.zps;
  dp.fp_values = p.fp_values;
  dp.out = out;
  dp.n = n;
  dp.nb = nb;
  return launch_staged(f, d, p, dp, static_cast<cudaStream_t>(stream)) == cudaSuccess ? QR_OK : QR_ERR_CUDA;
}
