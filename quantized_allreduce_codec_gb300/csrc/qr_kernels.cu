// qr_kernels.cu -- kernel instantiations and launchers for ONE format,
// selected at compile time with -DQR_FMT=<n> (the build compiles this file
// once per format, in parallel).
#include <atomic>

#include "qr_launch.h"

#ifndef QR_FMT
#error "compile with -DQR_FMT=<format number>"
#endif

#define QR_CAT2(a, b) a##b
#define QR_CAT(a, b) QR_CAT2(a, b)

namespace qr {
namespace {

constexpr int kMaxDevices = 64;

// Launch with programmatic stream serialization: the kernel may become
// resident while the previous kernel in the stream drains; it waits for that
// kernel's completion itself (wait_prior_grid) before touching memory.
template <typename Params>
cudaError_t launch_overlapped(void (*kern)(Params), dim3 grid, unsigned block, size_t smem, cudaStream_t s,
                              const Params& p) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(block);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, p);
}

// CTAs of `kern` that are resident on the current device at once (SMs x
// CTAs per SM at this block size and shared memory), computed once per
// device; grid-stride kernels are launched with at most this many, so every
// CTA starts at once and none waits for a second wave.  The cache is one
// atomic word per device: a thread sees either 0 (and computes the same
// value itself) or the complete value, never a half-written one.
template <typename Params>
cudaError_t resident_ctas(void (*kern)(Params), int threads, int smem, std::atomic<unsigned long long>* cache,
                          unsigned long long* out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  unsigned long long v = cache[dev].load(std::memory_order_acquire);
  if (v == 0) {
    int sms = 0, occ = 0;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, threads, smem);
    if (e != cudaSuccess) return e;
    v = static_cast<unsigned long long>(sms) * static_cast<unsigned long long>(occ > 0 ? occ : 1);
    cache[dev].store(v, std::memory_order_release);
  }
  *out = v;
  return cudaSuccess;
}

template <int F, int D, int M, int WS, int CW>
cudaError_t launch_pipe_w(const PipeParams& p, cudaStream_t s) {
  // Resident CTAs of this instantiation on each device, computed once per
  // device after its shared-memory limit is raised (resident_ctas' atomic
  // cache: the attribute is set before the value is published).
  static std::atomic<unsigned long long> cap[kMaxDevices];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  auto kern = qr_pipeline_kernel<F, D, M, WS, CW>;
  constexpr int kSmem = kSmemBytesOf<M, CW>;
  if (cap[dev].load(std::memory_order_acquire) == 0) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
    if (e != cudaSuccess) return e;
  }
  unsigned long long max_grid = 0;
  e = resident_ctas(kern, Tile<CW>::threads, kSmem, cap, &max_grid);
  if (e != cudaSuccess) return e;
  const unsigned long long ntiles = (p.n + Tile<CW>::elems - 1) / Tile<CW>::elems;
  const unsigned grid = static_cast<unsigned>(ntiles < max_grid ? ntiles : max_grid);
  return launch_overlapped(kern, grid, Tile<CW>::threads, kSmem, s, p);
}

// The rank count is a compile-time constant in every instantiation (W is
// one of 1, 2, 4, 8; encode-only runs one rank), except that the two-stage
// kernel at W = 8 runs the kernel's runtime rank loop (kW8Of = 0): its
// unrolled eight-rank body plus the requantization measured 1.5-3 % slower
// on GB300 than the one-rank loop body, while the one-stage kernel at W = 8
// is 1-2 % faster unrolled.
template <int F, int D, int M>
constexpr int kW8Of = M == MODE_AR2 ? 0 : 8;

// Narrow tiles (CW = 4) are built for W <= 4 only: at W = 8 they measured
// slower from 16 MiB per rank up, and below that the direct kernel serves
// W = 8; a W = 8 call asked for narrow tiles gets wide ones.
template <int F, int D, int M, int CW>
cudaError_t launch_pipe(const PipeParams& p, cudaStream_t s) {
  if constexpr (M == MODE_ENCODE) {
    return launch_pipe_w<F, D, M, 1, CW>(p, s);
  } else {
    switch (p.W) {
      case 1: return launch_pipe_w<F, D, M, 1, CW>(p, s);
      case 2: return launch_pipe_w<F, D, M, 2, CW>(p, s);
      case 4: return launch_pipe_w<F, D, M, 4, CW>(p, s);
      case 8: return launch_pipe_w<F, D, M, kW8Of<F, D, M>, kWideTile>(p, s);
      default: return cudaErrorInvalidValue;
    }
  }
}

template <int F, int D, int M>
cudaError_t launch_pipe_cw(int cw, const PipeParams& p, cudaStream_t s) {
  return cw == kNarrowTile ? launch_pipe<F, D, M, kNarrowTile>(p, s) : launch_pipe<F, D, M, kWideTile>(p, s);
}

// The direct kernel at W = 8 gets one CTA per 256 chunks, so each warp makes
// one pass (eight ranks' loads, the fold, the stores) and new CTAs start as
// earlier ones retire: on GB300 3-5 % faster from 4 MiB per rank up than a
// grid of resident CTAs looping over the message.  At W = 2 and 4 the
// resident grid measured as fast or faster (up to 5 % at 128 MiB) and stays.
// The direct path's kernel: for the W = 2 and W = 4 calls (one- and
// two-stage) of the integer formats the block kernel (one thread per block)
// from kBlockMinElemsOf elements per rank up, else the four-lanes-per-block
// direct kernel.  Below those sizes the block kernel has too few threads: at W = 4,
// 4 KiB-4 MiB per rank, it measured 0.3-0.8 us slower per call; the sizes are
// the ones that minimise the summed relative excess over the selection
// sweep's W = 2 and W = 4 two-stage integer shapes.
template <int F, int M, int WS>
constexpr bool kBlockKernelOf = (WS == 2 || WS == 4) && M != MODE_ENCODE && FmtInfo<F>::quant && !FmtInfo<F>::fp8;
template <int WS>
constexpr unsigned long long kBlockMinElemsOf = WS == 2 ? (3ull << 20) : (4ull << 20);

template <int F, int D, int M, int WS>
cudaError_t launch_dir_w(const PipeParams& p, cudaStream_t s) {
  if constexpr (kBlockKernelOf<F, M, WS>) {
    if (p.n >= kBlockMinElemsOf<WS>) {  // one CTA per kBlockThreads blocks, one pass
      const unsigned long long g = (p.nb + kBlockThreads - 1) / kBlockThreads;  // at most 2^24
      return launch_overlapped(qr_block_kernel<F, D, M, WS>, static_cast<unsigned>(g), kBlockThreads, 0, s, p);
    }
  }
  {
    const unsigned long long want = (p.nb * 4 + kDirectThreads - 1) / kDirectThreads;  // at most 2^25
    if constexpr (WS == 8) {
      return launch_overlapped(qr_direct_kernel<F, D, M, WS>, static_cast<unsigned>(want), kDirectThreads, 0, s, p);
    } else {
      static std::atomic<unsigned long long> cap[kMaxDevices];
      unsigned long long max_grid = 0;
      cudaError_t e = resident_ctas(qr_direct_kernel<F, D, M, WS>, kDirectThreads, 0, cap, &max_grid);
      if (e != cudaSuccess) return e;
      const unsigned grid = static_cast<unsigned>(want < max_grid ? want : max_grid);
      return launch_overlapped(qr_direct_kernel<F, D, M, WS>, grid, kDirectThreads, 0, s, p);
    }
  }
}

// The direct path's encoder (qr_quantize): one CTA per 256 blocks, one pass.
template <int F, int D>
cudaError_t launch_enc(const PipeParams& p, cudaStream_t s) {
  const unsigned long long grid = (p.nb + kEncodeBlocksPerCta - 1) / kEncodeBlocksPerCta;  // at most 2^23
  return launch_overlapped(qr_encode_kernel<F, D>, static_cast<unsigned>(grid), kEncodeThreads, 0, s, p);
}

template <int F, int D, int M>
cudaError_t launch_dir(const PipeParams& p, cudaStream_t s) {
  if constexpr (M == MODE_ENCODE) {
    return launch_enc<F, D>(p, s);
  } else {
    switch (p.W) {
      case 1: return launch_dir_w<F, D, M, 1>(p, s);
      case 2: return launch_dir_w<F, D, M, 2>(p, s);
      case 4: return launch_dir_w<F, D, M, 4>(p, s);
      case 8: return launch_dir_w<F, D, M, 8>(p, s);
      default: return cudaErrorInvalidValue;
    }
  }
}

// The decoder gets one CTA per kDecodeThreads x kDecodeUnroll chunks, so each
// thread makes one pass (its loads issued together, then its stores) and
// the hardware starts new CTAs as earlier ones retire; on GB300 this was 3-7 %
// faster than a grid of resident CTAs looping over the message, whose threads
// drain their loads between iterations.  (At most 2^36 / 8 / 1024 CTAs.)
template <int F, int D>
cudaError_t launch_dec(const DecodeParams& p, cudaStream_t s) {
  const unsigned long long per_cta = (unsigned long long)kDecodeThreads * kDecodeUnroll;
  const unsigned long long grid = (p.n / 8 + per_cta - 1) / per_cta;
  return launch_overlapped(qr_decode_kernel<F, D>, static_cast<unsigned>(grid), kDecodeThreads, 0, s, p);
}

// The staged kernels run one pass each (new CTAs start as earlier ones
// retire): the scatter-encoder one thread per (rank, block), rank =
// blockIdx.y; the owner reduction one thread per block with its rank loop
// unrolled for the compile-time W (kOwnerWs).  On GB300, W = 8 Q4 at 128 MiB
// per rank: 319 -> 294 us against one thread looping over the ranks in both
// kernels (the scatter 9 % faster, the unrolled owner 10 %).
template <int W>
constexpr int kOwnerWs = W == 1 ? 0 : W;

template <int F, int D, int WS>
cudaError_t launch_stg_w(const StagedParams& p, const DecodeParams& dp, cudaStream_t s) {
  const unsigned blocks = static_cast<unsigned>((p.nb + kStagedThreads - 1) / kStagedThreads);  // at most 2^23
  cudaError_t e = launch_overlapped(qr_scatter_encode_kernel<F, D>, dim3(blocks, WS), kStagedThreads, 0, s, p);
  if (e != cudaSuccess) return e;
  e = launch_overlapped(qr_owner_reduce_kernel<F, D, kOwnerWs<WS>>, dim3(blocks), kStagedThreads, 0, s, p);
  if (e != cudaSuccess) return e;
  return launch_dec<F, D>(dp, s);
}

template <int F, int D>
cudaError_t launch_stg(const StagedParams& p, const DecodeParams& dp, cudaStream_t s) {
  switch (p.W) {
    case 1: return launch_stg_w<F, D, 1>(p, dp, s);
    case 2: return launch_stg_w<F, D, 2>(p, dp, s);
    case 4: return launch_stg_w<F, D, 4>(p, dp, s);
    default: return launch_stg_w<F, D, 8>(p, dp, s);
  }
}

}  // namespace

cudaError_t QR_CAT(launch_staged_fmt_, QR_FMT)(int dt, const StagedParams& p, const DecodeParams& dp, cudaStream_t s) {
  constexpr int F = QR_FMT;
  if (dt == DT_F16) return launch_stg<F, DT_F16>(p, dp, s);
  return launch_stg<F, DT_BF16>(p, dp, s);
}

cudaError_t QR_CAT(launch_pipeline_fmt_, QR_FMT)(int dt, int mode, int cw, const PipeParams& p, cudaStream_t s) {
  constexpr int F = QR_FMT;
  if (dt == DT_BF16_AS_F16) {  // allreduce modes only
    if (mode == MODE_AR1) return launch_pipe_cw<F, DT_BF16_AS_F16, MODE_AR1>(cw, p, s);
    if (mode == MODE_AR2) return launch_pipe_cw<F, DT_BF16_AS_F16, MODE_AR2>(cw, p, s);
    return cudaErrorInvalidValue;
  }
  if (dt == DT_F16) {
    if (mode == MODE_ENCODE) return launch_pipe_cw<F, DT_F16, MODE_ENCODE>(cw, p, s);
    if (mode == MODE_AR1) return launch_pipe_cw<F, DT_F16, MODE_AR1>(cw, p, s);
    return launch_pipe_cw<F, DT_F16, MODE_AR2>(cw, p, s);
  }
  if (mode == MODE_ENCODE) return launch_pipe_cw<F, DT_BF16, MODE_ENCODE>(cw, p, s);
  if (mode == MODE_AR1) return launch_pipe_cw<F, DT_BF16, MODE_AR1>(cw, p, s);
  return launch_pipe_cw<F, DT_BF16, MODE_AR2>(cw, p, s);
}

cudaError_t QR_CAT(launch_direct_fmt_, QR_FMT)(int dt, int mode, const PipeParams& p, cudaStream_t s) {
  constexpr int F = QR_FMT;
  if (dt == DT_BF16_AS_F16) {  // allreduce modes only
    if (mode == MODE_AR1) return launch_dir<F, DT_BF16_AS_F16, MODE_AR1>(p, s);
    if (mode == MODE_AR2) return launch_dir<F, DT_BF16_AS_F16, MODE_AR2>(p, s);
    return cudaErrorInvalidValue;
  }
  if (dt == DT_F16) {
    if (mode == MODE_ENCODE) return launch_dir<F, DT_F16, MODE_ENCODE>(p, s);
    if (mode == MODE_AR1) return launch_dir<F, DT_F16, MODE_AR1>(p, s);
    return launch_dir<F, DT_F16, MODE_AR2>(p, s);
  }
  if (mode == MODE_ENCODE) return launch_dir<F, DT_BF16, MODE_ENCODE>(p, s);
  if (mode == MODE_AR1) return launch_dir<F, DT_BF16, MODE_AR1>(p, s);
  return launch_dir<F, DT_BF16, MODE_AR2>(p, s);
}

cudaError_t QR_CAT(launch_decode_fmt_, QR_FMT)(int dt, const DecodeParams& p, cudaStream_t s) {
  constexpr int F = QR_FMT;
  if (dt == DT_F16) return launch_dec<F, DT_F16>(p, s);
  return launch_dec<F, DT_BF16>(p, s);
}

}  // namespace qr
