// qr_launch.h -- internal interface between the C-ABI layer (qr_api.cu) and
// the per-format kernel translation units (qr_kernels.cu, built once per
// format with -DQR_FMT=<n>).
#pragma once

#include <cuda_runtime.h>

#include "qr.h"
#include "qr_device.cuh"
#include "qr_staged.cuh"

namespace qr {

// Launch the pipeline kernel (cw consumer warps per CTA: kWideTile or
// kNarrowTile) or the direct (small-message) kernel (encode / one-stage /
// two-stage) of format F for dtype dt, or the decode kernel; grids sized for
// the current device.
#define QR_DECLARE_FMT(N)                                                                           \
  cudaError_t launch_pipeline_fmt_##N(int dt, int mode, int cw, const PipeParams& p, cudaStream_t s); \
  cudaError_t launch_direct_fmt_##N(int dt, int mode, const PipeParams& p, cudaStream_t s);   \
  cudaError_t launch_decode_fmt_##N(int dt, const DecodeParams& p, cudaStream_t s);            \
  cudaError_t launch_staged_fmt_##N(int dt, const StagedParams& p, const DecodeParams& dp, cudaStream_t s);
QR_DECLARE_FMT(0)
QR_DECLARE_FMT(1)
QR_DECLARE_FMT(2)
QR_DECLARE_FMT(3)
QR_DECLARE_FMT(4)
QR_DECLARE_FMT(5)
QR_DECLARE_FMT(6)
#undef QR_DECLARE_FMT

// Device error flags word (defined in qr_api.cu).
unsigned* device_error_word();

// The staged two-stage allreduce (qr_allreduce_staged and
// qr_allreduce_staged_noalloc share these, so both use one slot geometry
// and one encoded layout).  staged_check_args: dtype, format, W and n, in
// that order.  staged_check_buffers (n > 0): every input non-NULL, then
// 16-byte alignment, then no overlap among the inputs, out, wire and (when
// not NULL) the caller's stage-1 buffer of qr_stage1_bytes(W, fmt, n) bytes.
// staged_launch: the three kernels on `s`, stage 1 in `stage1`, which must
// hold qr_stage1_bytes(W, fmt, n) bytes.
qr_status staged_check_args(int W, int dt, int fmt, size_t n);
qr_status staged_check_buffers(int W, int fmt, const void* const* inputs, size_t n, const void* out,
                               const void* wire, const void* stage1);
qr_status staged_launch(int W, int dt, int fmt, const void* const* inputs, size_t n, void* out, void* wire,
                        uint8_t* stage1, cudaStream_t s);

}  // namespace qr
