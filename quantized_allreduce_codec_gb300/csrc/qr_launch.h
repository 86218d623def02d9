// qr_launch.h -- internal interface between the C-ABI layer (qr_api.cu) and
// the per-format kernel translation units (qr_kernels.cu, built once per
// format with -DQR_FMT=<n>).
#pragma once

#include <cuda_runtime.h>

#include "qr_device.cuh"
#include "qr_staged.cuh"

namespace qr {

// Launch the pipeline kernel or the direct (small-message) kernel (encode /
// one-stage / two-stage) of format F for dtype dt, or the decode kernel;
// grids sized for the current device.
#define QR_DECLARE_FMT(N)                                                                   \
  cudaError_t launch_pipeline_fmt_##N(int dt, int mode, const PipeParams& p, cudaStream_t s); \
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

}  // namespace qr
