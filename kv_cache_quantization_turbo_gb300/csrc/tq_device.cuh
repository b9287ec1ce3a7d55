// Device helpers shared by the encode, dequantize and decode kernels.
#pragma once

#include <cstdint>

#include <cuda_fp16.h>

#include "tq_internal.h"

namespace tq {

constexpr unsigned kFull = 0xffffffffu;

// sqrt(pi/2): E[sign(g.r) g] = sqrt(2/pi) r/||r|| for g ~ N(0, I), so the
// residual inner product estimate is ||r|| sqrt(pi/2)/m <S q, sign(S r)>.
constexpr float kSqrtHalfPi = 1.2533141373155002512f;

template <int D>
__device__ __forceinline__ constexpr float inv_sqrt_dim() {
  return D == 64 ? 0.125f : D == 128 ? 0.08838834764831844055f : 0.0625f;
}

// Orthonormal Walsh-Hadamard transform of one d-vector held by a warp: lane l
// owns the E = D/32 consecutive coordinates [E*l, E*l + E) in x[].  Butterfly
// (a, b) -> (a + b, a - b) over strides 1, 2, ..., D/2 gives the natural
// (Sylvester) order; strides below E stay in registers, the others pair lane
// l with lane l ^ (stride / E).  The result is scaled by 1/sqrt(D).
template <int D>
__device__ __forceinline__ void warp_wht(float (&x)[D / 32], int lane) {
  constexpr int E = D / 32;
#pragma unroll
  for (int s = 1; s < E; s <<= 1) {
#pragma unroll
    for (int i = 0; i < E; ++i) {
      if ((i & s) == 0) {
        const float a = x[i], b = x[i + s];
        x[i] = a + b;
        x[i + s] = a - b;
      }
    }
  }
#pragma unroll
  for (int m = 1; m < 32; m <<= 1) {
    const bool upper = (lane & m) != 0;
#pragma unroll
    for (int i = 0; i < E; ++i) {
      const float o = __shfl_xor_sync(kFull, x[i], m);
      x[i] = upper ? (o - x[i]) : (x[i] + o);
    }
  }
  const float sc = inv_sqrt_dim<D>();
#pragma unroll
  for (int i = 0; i < E; ++i) x[i] *= sc;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int m = 16; m > 0; m >>= 1) v += __shfl_xor_sync(kFull, v, m);
  return v;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int m = 16; m > 0; m >>= 1) v = fmaxf(v, __shfl_xor_sync(kFull, v, m));
  return v;
}

// Programmatic dependent launch.  A kernel launched with launch_pdl may start while the kernel
// before it in the stream is still running, once every CTA of that kernel has called
// pdl_launch_dependents (or exited); before it reads anything that kernel writes it calls
// pdl_wait, which returns when that kernel has completed and its writes are visible.  Both are
// no-ops for kernels launched the ordinary way.
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

template <class... P, class... A>
cudaError_t launch_pdl(void (*kern)(P...), dim3 grid, dim3 block, size_t smem, cudaStream_t s, A&&... args) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<A&&>(args)...);
}

// Index of vector (layer, slot, head) in a view, or -1 if the slot is outside
// the layer's pages.
__device__ __forceinline__ long long view_vector_index(const DevView& v, int layer, long long slot, int head) {
  const long long cap = v.num_pages * (long long)v.page_size;
  if (slot < 0 || slot >= cap) return -1;
  const long long page = slot / v.page_size;
  const long long p = slot - page * v.page_size;
  return (((long long)layer * v.num_pages + page) * v.H + head) * v.page_size + p;
}

// Code of coordinate i in a little-endian stream of w-bit codes.
__device__ __forceinline__ uint32_t stream_code(const uint32_t* words, int i, int w) {
  const int bit = i * w;
  const int k = bit >> 5, sh = bit & 31;
  uint32_t v = words[k] >> sh;
  if (sh + w > 32) v |= words[k + 1] << (32 - sh);
  return v & ((1u << w) - 1u);
}

// Packs D w-bit codes (one byte each, codes[i] for coordinate i, in shared
// memory) into the little-endian stream and stores its D*w/32 words; lane j
// builds word j.  D*w/32 <= 32 for D <= 256 and w <= 4.
template <int D>
__device__ __forceinline__ void warp_pack_store(const uint8_t* codes, int w, uint32_t* dst, int lane) {
  const int nwords = D * w / 32;
  if (lane < nwords) {
    const int b0 = lane * 32;
    uint32_t word = 0;
    int i = b0 / w;
    for (; i * w < b0 + 32 && i < D; ++i) {
      const int off = i * w - b0;
      const uint32_t c = codes[i];
      word |= off >= 0 ? (c << off) : (c >> (-off));
    }
    dst[lane] = word;
  }
}

}  // namespace tq
