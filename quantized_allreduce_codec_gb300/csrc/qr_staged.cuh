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
  float one;                      // 1.0f; see biased_code2
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

// Owner of block blk: the number of owner starts k*chunk_nb (k >= 1) at or
// below it (W - 1 comparisons; no division).
__device__ __forceinline__ unsigned long long owner_of(unsigned long long blk, unsigned long long chunk_nb, int W) {
  unsigned long long j = 0;
#pragma unroll
  for (int k = 1; k < 8; ++k)
    if (k < W && blk >= static_cast<unsigned long long>(k) * chunk_nb) ++j;
  return j;
}

constexpr int kStagedThreads = 256;

// Block scale and clamp-free flag of one block held as raw 16-bit words
// (invalid chunks zeroed), as in the pipeline kernel's stage 1.
template <int F, int D>
__device__ __forceinline__ BlockScale raw_block_scale(const uint4 (&raw)[4], int nvalid, bool& fast) {
  if (FmtInfo<F>::asym) {
    float m, M;
    raw_minmax<D>(raw, 0, nvalid, m, M);
    const BlockScale b = scale_from_minmax<F>(m, M);
    fast = clamp_free<F>(b, m, M);
    return b;
  }
  const float a = raw_absmax<D>(raw);
  const BlockScale b = scale_from_absmax<F>(a);
  fast = FmtInfo<F>::fp8 ? true : clamp_free<F>(b, 0.0f, a);
  return b;
}

template <int F>
__device__ __forceinline__ BlockScale f32_block_scale(const float (&x)[32], int nvalid, bool& fast) {
  if (FmtInfo<F>::asym) {
    float m, M;
    f32_minmax(x, 0, nvalid, m, M);
    const BlockScale b = scale_from_minmax<F>(m, M);
    fast = clamp_free<F>(b, m, M);
    return b;
  }
  const float a = f32_absmax(x);
  const BlockScale b = scale_from_absmax<F>(a);
  fast = FmtInfo<F>::fp8 ? true : clamp_free<F>(b, 0.0f, a);
  return b;
}

// Encode the four chunks of a block and store codes / scale / zero-point into
// an encoded region (codes at codes + blk*cb, scale at scales[blk]); chunk(k,
// x) puts chunk k's eight binary32 values in x.  The block's code bytes are
// assembled in registers and written with the widest aligned stores (32 B:
// two 16-byte stores; 16 B: one; Q6's 24 B: three 8-byte stores).
template <int F, typename ChunkFn>
__device__ __forceinline__ void encode_store_block(ChunkFn&& chunk, const BlockScale& b, float one, bool fast,
                                                   int nvalid, uint8_t* codes, uint16_t* scales, uint16_t* zps,
                                                   unsigned long long blk) {
  uint32_t pk[4][2];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    float x[8], dec[8];
    pk[k][0] = pk[k][1] = 0u;
    chunk(k, x);
    if (fast)
      encode8<F, true>(x, b, one, dec, pk[k]);
    else
      encode8<F, false>(x, b, one, dec, pk[k]);
    if (FmtInfo<F>::asym && k >= nvalid) pk[k][0] = pk[k][1] = 0u;  // pad codes are 0
  }
  uint8_t* cp = codes + blk * FmtInfo<F>::code_bytes;
  if (FmtInfo<F>::bits == 8) {
    reinterpret_cast<uint4*>(cp)[0] = make_uint4(pk[0][0], pk[0][1], pk[1][0], pk[1][1]);
    reinterpret_cast<uint4*>(cp)[1] = make_uint4(pk[2][0], pk[2][1], pk[3][0], pk[3][1]);
  } else if (FmtInfo<F>::bits == 4) {
    reinterpret_cast<uint4*>(cp)[0] = make_uint4(pk[0][0], pk[1][0], pk[2][0], pk[3][0]);
  } else {  // four 48-bit pieces -> 192-bit little-endian stream
    const uint32_t w0 = pk[0][0], w1 = (pk[0][1] & 0xFFFFu) | (pk[1][0] << 16);
    const uint32_t w2 = (pk[1][0] >> 16) | (pk[1][1] << 16), w3 = pk[2][0];
    const uint32_t w4 = (pk[2][1] & 0xFFFFu) | (pk[3][0] << 16), w5 = (pk[3][0] >> 16) | (pk[3][1] << 16);
    uint2* c2 = reinterpret_cast<uint2*>(cp);  // 8-byte aligned: blk*24
    c2[0] = make_uint2(w0, w1);
    c2[1] = make_uint2(w2, w3);
    c2[2] = make_uint2(w4, w5);
  }
  scales[blk] = b.s_bits;
  if (FmtInfo<F>::asym) zps[blk] = b.z_bits;
}

// Number of valid 8-element chunks of block blk: 4 unless the block is the
// message's ragged last one.  FULL asserts that blk lies wholly inside.
template <bool FULL>
__device__ __forceinline__ int valid_chunks(unsigned long long n, unsigned long long blk) {
  if constexpr (FULL) return 4;
  const unsigned long long rem = n - blk * 32;
  return rem >= 32 ? 4 : static_cast<int>(rem / 8);
}

// Kernel 1: one thread per (rank, block) -- rank blockIdx.y, block
// blockIdx.x * kStagedThreads + threadIdx.x -- in one pass: load the block's
// 64 bytes, encode it and write it into slot (owner, rank) at the owner's
// local block index.  No loop over ranks: the W ranks' blocks are W times as
// many independent threads, each holding one block's loads.
template <int F, int D, bool FULL>
__device__ __forceinline__ void scatter_block(const StagedParams& p, int r, unsigned long long blk) {
  const int nvalid = valid_chunks<FULL>(p.n, blk);
  const unsigned long long j = owner_of(blk, p.chunk_nb, p.W);
  const unsigned long long local = blk - j * p.chunk_nb;
  uint8_t* slot = p.stage1 + (j * p.W + r) * p.slot_bytes;
  const uint4* src = reinterpret_cast<const uint4*>(p.in[r]) + blk * 4;
  uint4 raw[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) raw[k] = (FULL || k < nvalid) ? __ldg(src + k) : make_uint4(0u, 0u, 0u, 0u);
  if constexpr (!FmtInfo<F>::quant) {
#pragma unroll
    for (int k = 0; k < 4; ++k)
      if (FULL || k < nvalid) reinterpret_cast<uint4*>(slot + local * 64)[k] = raw[k];
  } else {
    bool fast;
    const BlockScale b = raw_block_scale<F, D>(raw, nvalid, fast);
    encode_store_block<F>([&](int k, float* x) { widen8<D>(raw[k], x); }, b, p.one, fast, nvalid, slot,
                          reinterpret_cast<uint16_t*>(slot + slot_scales_off<F>(p.chunk_nb)),
                          reinterpret_cast<uint16_t*>(slot + slot_zps_off<F>(p.chunk_nb)), local);
  }
}

template <int F, int D>
__global__ void __launch_bounds__(kStagedThreads) qr_scatter_encode_kernel(const __grid_constant__ StagedParams p) {
  wait_prior_grid();
  allow_next_grid();
  const int r = static_cast<int>(blockIdx.y);
  const unsigned long long blk = static_cast<unsigned long long>(blockIdx.x) * kStagedThreads + threadIdx.x;
  if (blk < p.n / 32)
    scatter_block<F, D, true>(p, r, blk);
  else if (blk < p.nb)
    scatter_block<F, D, false>(p, r, blk);
}

// Calls f(r) for the ranks r = 0 .. W-1 in order: fully unrolled when the
// rank count WS is a compile-time constant, a runtime loop when WS is 0.
template <int WS, typename Fn>
__device__ __forceinline__ void for_ranks(int W, Fn&& f) {
  if constexpr (WS > 0) {
#pragma unroll
    for (int r = 0; r < WS; ++r) f(r);
  } else {
    for (int r = 0; r < W; ++r) f(r);
  }
}

// Code words of chunk k of a block whose code bytes are in cw (up to 32 bytes
// as eight 32-bit words).
template <int F>
__device__ __forceinline__ uint2 chunk_code_words(const uint32_t (&cw)[8], int k) {
  if (FmtInfo<F>::bits == 8) return make_uint2(cw[2 * k], cw[2 * k + 1]);
  if (FmtInfo<F>::bits == 4) return make_uint2(cw[k], 0u);
  // 6 bits: chunk k's 48 bits start at bit 48k of the block's stream
  const int bit = 48 * k, w0 = bit >> 5, sh = bit & 31;
  const uint32_t lo = __funnelshift_r(cw[w0], cw[w0 + 1], sh);
  const uint32_t hi = __funnelshift_r(cw[w0 + 1], w0 + 2 < 8 ? cw[w0 + 2] : 0u, sh) & 0xFFFFu;
  return make_uint2(lo, hi);
}

// A block's code words (up to 32 bytes), scale and zero-point from a slot.
template <int F>
__device__ __forceinline__ void load_slot_block(const uint8_t* slot, unsigned long long chunk_nb,
                                                unsigned long long local, uint32_t (&cw)[8], uint16_t& s_bits,
                                                uint16_t& z_bits) {
  const uint8_t* cp = slot + local * FmtInfo<F>::code_bytes;
  if (FmtInfo<F>::bits == 8) {
    const uint4 a0 = __ldg(reinterpret_cast<const uint4*>(cp)), a1 = __ldg(reinterpret_cast<const uint4*>(cp) + 1);
    cw[0] = a0.x; cw[1] = a0.y; cw[2] = a0.z; cw[3] = a0.w;
    cw[4] = a1.x; cw[5] = a1.y; cw[6] = a1.z; cw[7] = a1.w;
  } else if (FmtInfo<F>::bits == 4) {
    const uint4 a0 = __ldg(reinterpret_cast<const uint4*>(cp));
    cw[0] = a0.x; cw[1] = a0.y; cw[2] = a0.z; cw[3] = a0.w;
    cw[4] = cw[5] = cw[6] = cw[7] = 0u;
  } else {  // 24 bytes at an 8-byte aligned offset
    const uint2* c2 = reinterpret_cast<const uint2*>(cp);
    const uint2 a0 = __ldg(c2), a1 = __ldg(c2 + 1), a2 = __ldg(c2 + 2);
    cw[0] = a0.x; cw[1] = a0.y; cw[2] = a1.x; cw[3] = a1.y; cw[4] = a2.x; cw[5] = a2.y;
    cw[6] = cw[7] = 0u;
  }
  s_bits = __ldg(reinterpret_cast<const unsigned short*>(slot + slot_scales_off<F>(chunk_nb)) + local);
  z_bits = FmtInfo<F>::asym ? __ldg(reinterpret_cast<const unsigned short*>(slot + slot_zps_off<F>(chunk_nb)) + local)
                            : static_cast<uint16_t>(0);
}

// Kernel 2: one thread per block; the owner decodes the block from its W
// source slots (each rank's loaded one rank ahead), sums them in rank order
// and requantizes into the payload.  reduce_block is one block's work; WS is
// the rank count when it is known at compile time (2, 4, 8) or 0, and FULL
// (used only with a known WS) that the block is complete.
template <int F, int D, int WS, bool FULL>
__device__ __forceinline__ void reduce_block(const StagedParams& p, unsigned long long blk) {
  const int W = WS ? WS : p.W;
    const int nvalid = valid_chunks<FULL>(p.n, blk);
    const unsigned long long j = owner_of(blk, p.chunk_nb, W);
    const unsigned long long local = blk - j * p.chunk_nb;
    float acc[32];
    if constexpr (!FmtInfo<F>::quant) {
      for_ranks<WS>(W, [&](int r) {
        const uint4* src = reinterpret_cast<const uint4*>(p.stage1 + (j * W + r) * p.slot_bytes + local * 64);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          float y[8];
          widen8<D>(k < nvalid ? __ldg(src + k) : make_uint4(0u, 0u, 0u, 0u), y);
#pragma unroll
          for (int i = 0; i < 8; ++i) acc[8 * k + i] = (r == 0) ? y[i] : __fadd_rn(acc[8 * k + i], y[i]);
        }
      });
      uint4* dst = reinterpret_cast<uint4*>(p.fp_values) + blk * 4;
#pragma unroll
      for (int k = 0; k < 4; ++k)
        if (k < nvalid) dst[k] = narrow8<D>(&acc[8 * k]);
    } else {
      uint32_t cw[8], ncw[8];  // this rank's and the next rank's code words
      uint16_t sb = 0, zb = 0, nsb = 0, nzb = 0;
      load_slot_block<F>(p.stage1 + j * W * p.slot_bytes, p.chunk_nb, local, ncw, nsb, nzb);
      for_ranks<WS>(W, [&](int r) {
#pragma unroll
        for (int i = 0; i < 8; ++i) cw[i] = ncw[i];
        sb = nsb;
        zb = nzb;
        if (r + 1 < W) load_slot_block<F>(p.stage1 + (j * W + r + 1) * p.slot_bytes, p.chunk_nb, local, ncw, nsb, nzb);
        BlockScale b;
        b.s = __half2float(__ushort_as_half(sb));
        b.z = FmtInfo<F>::asym ? __half2float(__ushort_as_half(zb)) : 0.0f;
        // same bits as the fused kernel: exact products, rank order
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          if (r == 0)
            unpack8_accumulate<F, true>(chunk_code_words<F>(cw, k), b, &acc[8 * k]);
          else
            unpack8_accumulate<F, false>(chunk_code_words<F>(cw, k), b, &acc[8 * k]);
        }
      });
      if (nvalid < 4 && !FmtInfo<F>::asym) {  // the symmetric statistic skips invalid chunks as zeros
#pragma unroll
        for (int k = 0; k < 4; ++k)
          if (k >= nvalid) {
#pragma unroll
            for (int i = 0; i < 8; ++i) acc[8 * k + i] = 0.0f;
          }
      }
      bool fast;
      const BlockScale b2 = f32_block_scale<F>(acc, nvalid, fast);
      encode_store_block<F>(
          [&](int k, float* x) {
#pragma unroll
            for (int i = 0; i < 8; ++i) x[i] = acc[8 * k + i];
          },
          b2, p.one, fast, nvalid, p.codes, p.scales, p.zps, blk);
    }
}

template <int F, int D, int WS>
__global__ void __launch_bounds__(kStagedThreads) qr_owner_reduce_kernel(const __grid_constant__ StagedParams p) {
  wait_prior_grid();
  allow_next_grid();
  const unsigned long long stride = (unsigned long long)gridDim.x * kStagedThreads;
  const unsigned long long nb_full = p.n / 32;
  for (unsigned long long blk = (unsigned long long)blockIdx.x * kStagedThreads + threadIdx.x; blk < p.nb;
       blk += stride) {
    if constexpr (WS > 0) {
      if (blk < nb_full)
        reduce_block<F, D, WS, true>(p, blk);
      else
        reduce_block<F, D, WS, false>(p, blk);
    } else {
      reduce_block<F, D, 0, false>(p, blk);
    }
  }
}

}  // namespace qr
