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

}  // namespace
}  // namespace qr

using namespace qr;

extern "C" qr_status qr_allreduce_staged_noalloc(int W, qr_dtype dt, qr_format fmt, const void* const* inputs,
                                                 size_t n, void* out, void* wire, void* stream) {
  const int f = static_cast<int>(fmt), d = static_cast<int>(dt);
  if (n && (!inputs || !out || !wire)) return QR_ERR_NULL;
  qr_status st = staged_check_args(W, d, f, n);
  if (st != QR_OK) return st;
  if (n == 0) return QR_OK;
  // qr_stage1_bytes is the size staged_launch lays the slots out in, so this
  // bound is exactly what the kernels write into the array
  if (qr_stage1_bytes(W, fmt, n) > kNoAllocScratchBytes) return QR_ERR_SCRATCH;
  st = staged_check_buffers(W, f, inputs, n, out, wire, nullptr);
  if (st != QR_OK) return st;
  uint8_t* scratch = scratch_address();
  if (!scratch) return QR_ERR_CUDA;
  return staged_launch(W, d, f, inputs, n, out, wire, scratch, static_cast<cudaStream_t>(stream));
}
