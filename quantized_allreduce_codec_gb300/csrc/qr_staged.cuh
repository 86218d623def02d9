// qr_staged.cuh -- the two-stage allreduce with its stage-1 exchange
// materialised: the structure a real multi-GPU quick allreduce has ("2stage"
// of vLLM PR #18473, "two shot" of vLLM PR #16804), emulated on one GPU.
//
//   kernel 1 (scatter-encode): every rank r encodes its message; block b
//     belongs to owner j = b / chunk_nb, and its codes go to owner j's
//     receive slot for source r in the stage-1 buffer;
//   kernel 2 (owner reduce): for each block, its owner decodes the W source
//     slots, accumulates in rank order (binary32) and requantizes the sum into
//     the stage-2 payload (the all-gather buffer, standard encoded layout);
//   kernel 3 (decode): the payload is decoded to the output (qr_dequantize).
//
// The arithmetic is the fused kernel's, operation for operation, so outputs
// and payloads are bit-identical; what differs is the traffic: the stage-1
// codes make a round trip through HBM and the work takes three launches.
//
// Stage-1 buffer layout: W x W slots, slot (j, r) at (j*W + r) * slot_bytes,
// each an encoded sub-message of chunk_nb blocks in structure-of-arrays form
// (codes[chunk_nb][cb] | scales[chunk_nb] | zps[chunk_nb]), padded to 16
// bytes; FP passthrough slots hold the chunk's values.
#pragma once

#include "qr_device.cuh"

namespace qr {

struct StagedParams {
  const void* in[8];
  int W;
  unsigned long long n, nb;
  unsigned long long chunk_nb;    // blocks per owner
  unsigned long long slot_bytes;  // bytes per (owner, source) slot
  uint8_t* stage1;                // W*W slots
  uint8_t* codes;                 // stage-2 payload regions (standard layout)
  uint16_t* scales;
  uint16_t* zps;
  uint16_t* fp_values;            // FP format: payload values
};

// Byte offsets of the regions of one slot.
template <int F>
__device__ __forceinline__ unsigned long long slot_scales_off(unsigned long long chunk_nb) {
  return chunk_nb * FmtInfo<F>::code_bytes;
}
template <int F>
__device__ __forceinline__ unsigned long long slot_zps_off(unsigned long long chunk_nb) {
  return chunk_nb * (FmtInfo<F>::code_bytes + 2);
}

// Kernel 1: one thread per (rank, 8-element chunk); four lanes per block.
template <int F, int D>
__global__ void __launch_bounds__(kDirectThreads) qr_scatter_encode_kernel(const __grid_constant__ StagedParams p) {
  const int lane = threadIdx.x & 31;
  const unsigned long long per_rank = p.nb * 4;  // chunk slots per rank (padded final block)
  const unsigned long long total = per_rank * p.W;
  const unsigned long long nchunks = p.n / 8;
  const unsigned long long stride = (unsigned long long)gridDim.x * kDirectThreads;
  for (unsigned long long base = (unsigned long long)blockIdx.x * kDirectThreads + (threadIdx.x & ~31u);
       base < total; base += stride) {
    const unsigned long long idx = base + lane;
    const bool live = idx < total;
    const int r = live ? static_cast<int>(idx / per_rank) : 0;
    const unsigned long long g = live ? idx - static_cast<unsigned long long>(r) * per_rank : 0;
    const bool valid = live && g < nchunks;
    const unsigned long long blk = g >> 2;
    const int c = static_cast<int>(g & 3);
    const unsigned long long j = blk / p.chunk_nb;
    const unsigned long long local = blk - j * p.chunk_nb;
    uint8_t* slot = p.stage1 + (j * p.W + r) * p.slot_bytes;

    uint4 raw = make_uint4(0u, 0u, 0u, 0u);
    if (valid) raw = reinterpret_cast<const uint4*>(p.in[r])[g];
    if constexpr (!FmtInfo<F>::quant) {
      if (valid) reinterpret_cast<uint4*>(slot + local * 64)[c] = raw;
    } else {
      bool fast;
      const BlockScale b = group_scale_raw<F, D>(raw, valid, fast);
      float x[8], dec[8];
      uint32_t packed[2] = {0u, 0u};
      widen8<D>(raw, x);
      if (fast)
        encode8<F, true>(x, b, dec, packed);
      else
        encode8<F, false>(x, b, dec, packed);
      if (!valid) packed[0] = packed[1] = 0u;  // pad codes are 0
      if (live) store_chunk_codes<F>(slot, local, c, packed);
      if (live && c == 0) {
        reinterpret_cast<uint16_t*>(slot + slot_scales_off<F>(p.chunk_nb))[local] = b.s_bits;
        if (FmtInfo<F>::asym) reinterpret_cast<uint16_t*>(slot + slot_zps_off<F>(p.chunk_nb))[local] = b.z_bits;
      }
    }
  }
}

// Kernel 2: one thread per 8-element chunk of the message; the owner of its
// block reduces the W source slots and requantizes into the payload.
template <int F, int D>
__global__ void __launch_bounds__(kDirectThreads) qr_owner_reduce_kernel(const __grid_constant__ StagedParams p) {
  const int lane = threadIdx.x & 31;
  const unsigned long long total = p.nb * 4;
  const unsigned long long nchunks = p.n / 8;
  const unsigned long long stride = (unsigned long long)gridDim.x * kDirectThreads;
  for (unsigned long long base = (unsigned long long)blockIdx.x * kDirectThreads + (threadIdx.x & ~31u);
       base < total; base += stride) {
    const unsigned long long g = base + lane;
    const bool in_block = g < total;
    const bool valid = g < nchunks;
    const unsigned long long blk = in_block ? (g >> 2) : 0;
    const int c = static_cast<int>(g & 3);
    const unsigned long long j = blk / p.chunk_nb;
    const unsigned long long local = blk - j * p.chunk_nb;

    float acc[8];
#pragma unroll
    for (int r = 0; r < 8; ++r) {
      if (r >= p.W) break;
      const uint8_t* slot = p.stage1 + (j * p.W + r) * p.slot_bytes;
      float y[8];
      if constexpr (!FmtInfo<F>::quant) {
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (valid) v = reinterpret_cast<const uint4*>(slot + local * 64)[c];
        widen8<D>(v, y);
      } else {
        BlockScale b;
        b.s = 0.0f;
        b.z = 0.0f;
        if (in_block) {
          b.s = __half2float(__ushort_as_half(reinterpret_cast<const uint16_t*>(slot + slot_scales_off<F>(p.chunk_nb))[local]));
          if (FmtInfo<F>::asym)
            b.z = __half2float(__ushort_as_half(reinterpret_cast<const uint16_t*>(slot + slot_zps_off<F>(p.chunk_nb))[local]));
          unpack8<F>(slot + local * FmtInfo<F>::code_bytes, c, b, y);
        } else {
#pragma unroll
          for (int i = 0; i < 8; ++i) y[i] = 0.0f;
        }
      }
      // decoded values are exact, so this add equals the fused kernel's FMA
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[i] = (r == 0) ? y[i] : __fadd_rn(acc[i], y[i]);
    }

    if constexpr (!FmtInfo<F>::quant) {
      if (valid) reinterpret_cast<uint4*>(p.fp_values)[g] = narrow8<D>(acc);
    } else {
      bool fast;
      const BlockScale b2 = group_scale_f32<F>(acc, valid, fast);
      float dec[8];
      uint32_t packed[2] = {0u, 0u};
      if (fast)
        encode8<F, true>(acc, b2, dec, packed);
      else
        encode8<F, false>(acc, b2, dec, packed);
      if (!valid) packed[0] = packed[1] = 0u;
      if (in_block) store_chunk_codes<F>(p.codes, blk, c, packed);
      if (in_block && c == 0) {
        p.scales[blk] = b2.s_bits;
        if (FmtInfo<F>::asym) p.zps[blk] = b2.z_bits;
      }
    }
  }
}

}  // namespace qr
