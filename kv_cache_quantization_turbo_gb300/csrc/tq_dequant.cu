// Dequantize kernel: stored vectors -> fp32 reconstruction in the original space.
//
// Turbo ("TurboQuant+ KV cache compression", Stage 1 and Stage 2):
//   x~ = diag(s) H ( n c[idx]  +  rnorm sqrt(pi/2)/d S^T (2 sigma - 1) ),
// the second term only for K formats with include_qjl (vector form of the
// QJL estimate).  q8_0: q * delta per block of 32.  min-max: q * scale + zero
// per group of 64 ("mac-code TurboQuant analysis", section 2.1).
// One warp per (slot, head); lane l owns coordinates [E l, E l + E), E = d/32.
#include <cuda_fp16.h>

#include "tq_device.cuh"

namespace tq {
namespace {

constexpr int kDqWarps = 4;

struct DqArgs {
  DevView view;
  DevTables tab;
  int layer;
  const long long* slots;
  long long slot_begin;
  int n;
  int include_qjl;
  float* out;
};

template <int D>
__global__ void __launch_bounds__(kDqWarps * 32) dequant_kernel(DqArgs a) {
  constexpr int E = D / 32;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  __shared__ uint32_t words_s[kDqWarps][D / 8];   // up to d*4 bits of codes per vector
  __shared__ float pm_s[kDqWarps][D];             // 2 sigma_j - 1
  const DevView& V = a.view;
  const long long item = (long long)blockIdx.x * kDqWarps + warp;  // (t, head), head fastest
  if (item >= (long long)a.n * V.H) return;                        // warp-uniform
  const int h = (int)(item % V.H);
  const long long t = item / V.H;
  const long long slot = a.slots ? a.slots[t] : a.slot_begin + t;
  const long long vid = view_vector_index(V, a.layer, slot, h);
  float* dst = a.out + item * D + E * lane;
  if (vid < 0) {
    if (lane == 0 && h == 0) atomicOr(a.tab.status, kFlagSlot);
#pragma unroll
    for (int e = 0; e < E; ++e) dst[e] = 0.f;
    return;
  }
  const unsigned char* pay = V.payload + vid * V.pay_bytes;
  const unsigned char* hdr = V.header + vid * V.hdr_bytes;
  float y[E];
  if (V.format == TQ_FMT_Q8_0) {
    const int8_t* q = reinterpret_cast<const int8_t*>(pay);
    const float delta = __half2float(reinterpret_cast<const __half*>(hdr)[(E * lane) / 32]);
#pragma unroll
    for (int e = 0; e < E; ++e) dst[e] = (float)q[E * lane + e] * delta;
    return;
  }
  const int nwords = V.pay_bytes / 4;
  for (int k = lane; k < nwords; k += 32) words_s[warp][k] = reinterpret_cast<const uint32_t*>(pay)[k];
  __syncwarp();
  if (V.format == TQ_FMT_MINMAX) {
    const __half2 sz = reinterpret_cast<const __half2*>(hdr)[(E * lane) / 64];
    const float sc = __low2float(sz), zr = __high2float(sz);
#pragma unroll
    for (int e = 0; e < E; ++e) {
      const float q = (float)stream_code(words_s[warp], E * lane + e, V.code_bits);
      dst[e] = fmaf(q, sc, zr);
    }
    return;
  }
  // turbo
  const int b = V.idx_bits;
  const float* cb = a.tab.centroids + (b - 1) * 8;
  const float n = __half2float(reinterpret_cast<const __half*>(hdr)[0]);
#pragma unroll
  for (int e = 0; e < E; ++e) {
    const uint32_t c = stream_code(words_s[warp], E * lane + e, V.code_bits);
    y[e] = n * cb[c & ((1u << b) - 1u)];
  }
  if (V.has_qjl && a.include_qjl) {
    const float rn = __half2float(reinterpret_cast<const __half*>(hdr)[1]);
    for (int j = lane; j < D; j += 32)
      pm_s[warp][j] = ((stream_code(words_s[warp], j, V.code_bits) >> b) & 1u) ? 1.f : -1.f;
    __syncwarp();
    float acc[E];
#pragma unroll
    for (int e = 0; e < E; ++e) acc[e] = 0.f;
    for (int j = 0; j < D; ++j) {
      const float pm = pm_s[warp][j];
#pragma unroll
      for (int e = 0; e < E; ++e) acc[e] = fmaf(__ldg(a.tab.S + j * D + E * lane + e), pm, acc[e]);
    }
    const float k = rn * kSqrtHalfPi / (float)D;
#pragma unroll
    for (int e = 0; e < E; ++e) y[e] = fmaf(k, acc[e], y[e]);
  }
  warp_wht<D>(y, lane);
#pragma unroll
  for (int e = 0; e < E; ++e) dst[e] = y[e] * (float)a.tab.signs[E * lane + e];
}

}  // namespace

cudaError_t launch_dequant(const DevTables& t, const DevView& view, int layer, const long long* slots,
                           long long slot_begin, int n, int include_qjl, float* out, cudaStream_t s) {
  DqArgs a{view, t, layer, slots, slot_begin, n, include_qjl, out};
  const long long items = (long long)n * view.H;
  const unsigned grid = (unsigned)((items + kDqWarps - 1) / kDqWarps);
  switch (view.d) {
    case 64: dequant_kernel<64><<<grid, kDqWarps * 32, 0, s>>>(a); break;
    case 128: dequant_kernel<128><<<grid, kDqWarps * 32, 0, s>>>(a); break;
    case 256: dequant_kernel<256><<<grid, kDqWarps * 32, 0, s>>>(a); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace tq
