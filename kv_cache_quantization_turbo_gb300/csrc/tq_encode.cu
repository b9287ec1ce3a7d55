// Encode kernels: fp16 K/V vectors -> stored codes + per-vector headers.
//
// Turbo formats ("TurboQuant+ KV cache compression", Stage 1 and Stage 2 step
// lists): norm, sign flip + Walsh-Hadamard rotation held in registers of one
// warp, Lloyd-Max index by boundary comparison; K adds the residual norm and
// the sign of each of the d random projections of the residual.
// q8_0 ("TurboQuant+ deep dive", section 2.1 absmax rule with n = 8, blocks of
// 32) and per-group min-max ("mac-code TurboQuant analysis", section 2.1) are
// the pages' baselines.
//
// Work decomposition
//   - one warp per vector for everything but the QJL projection; lane l holds
//     the E = d/32 consecutive coordinates [E l, E l + E);
//   - turbo K: a CTA encodes a batch of NV = 8192/d vectors: phase A (warps:
//     stage 1 and the residual r into shared memory), phase B (the whole CTA:
//     the d x d projection S r for every vector of the batch, each thread a
//     register tile of 8 vectors x 4 projections streaming S^T rows through
//     the L1 cache), phase C (warps: pack codes and store);
//   - grids are persistent: min(work, resident CTAs) CTAs loop over batches.
#include <cuda_fp16.h>

#include "tq_device.cuh"

namespace tq {
namespace {

enum EncKind { kTurboK = 0, kTurboV = 1, kQ8 = 2, kMinMax = 3 };

constexpr int kEncThreads = 256;
constexpr int kEncWarps = kEncThreads / 32;
constexpr int kVPT = 8;  // vectors per thread in the projection tile

template <int D>
struct EncShape {
  static constexpr int E = D / 32;
  static constexpr int JG = D / 4;                 // thread groups over projections
  static constexpr int VG = kEncThreads / JG;      // thread groups over vectors
  static constexpr int NV = VG * kVPT;             // vectors per batch (turbo K)
};

struct EncArgs {
  DevView view;
  DevTables tab;
  const __half* x;
  int layer_begin, n_layers, n_tokens;
  long long layer_stride, token_stride;
  const long long* slots;
  long long slot_begin;
  long long n_vectors;  // n_layers * n_tokens * H
};

// Global vector id -> (input layer, token, head) and the destination index
// in the view (-1 if the slot is out of range; the status word is flagged).
__device__ __forceinline__ long long enc_locate(const EncArgs& a, long long gv, const __half** src) {
  // vector counts stay below 2^32 (checked on the host): 32-bit division is enough
  const unsigned int H = (unsigned int)a.view.H, v32 = (unsigned int)gv;
  const unsigned int lt = v32 / H;
  const int h = (int)(v32 - lt * H);
  const unsigned int l32 = lt / (unsigned int)a.n_tokens;
  const int t = (int)(lt - l32 * (unsigned int)a.n_tokens);
  const int l = (int)l32;
  *src = a.x + l * a.layer_stride + t * a.token_stride + (long long)h * a.view.d;
  const long long slot = a.slots ? a.slots[t] : a.slot_begin + t;
  const long long v = view_vector_index(a.view, a.layer_begin + l, slot, h);
  if (v < 0 && h == 0) atomicOr(a.tab.status, kFlagSlot);
  return v;
}

template <int D>
__device__ __forceinline__ void load_vec(const __half* src, float (&x)[D / 32], int lane) {
  constexpr int E = D / 32;
  const __half* p = src + E * lane;
  if constexpr (E == 2) {
    const __half2 h = *reinterpret_cast<const __half2*>(p);
    x[0] = __low2float(h); x[1] = __high2float(h);
  } else if constexpr (E == 4) {
    const uint2 u = *reinterpret_cast<const uint2*>(p);
    const __half2 h0 = *reinterpret_cast<const __half2*>(&u.x), h1 = *reinterpret_cast<const __half2*>(&u.y);
    x[0] = __low2float(h0); x[1] = __high2float(h0); x[2] = __low2float(h1); x[3] = __high2float(h1);
  } else {
    const uint4 u = *reinterpret_cast<const uint4*>(p);
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const __half2 h = *reinterpret_cast<const __half2*>(&w[k]);
      x[2 * k] = __low2float(h); x[2 * k + 1] = __high2float(h);
    }
  }
}

// Stage 1 for one vector held by a warp: returns n and leaves y = H diag(s) x_hat in x.
template <int D>
__device__ __forceinline__ float stage1_rotate(float (&x)[D / 32], const int8_t* signs_s, int lane) {
  constexpr int E = D / 32;
  float ss = 0.f;
#pragma unroll
  for (int e = 0; e < E; ++e) ss = fmaf(x[e], x[e], ss);
  const float n = sqrtf(warp_sum(ss));
  const float inv = n > 0.f ? 1.0f / n : 0.f;
#pragma unroll
  for (int e = 0; e < E; ++e) x[e] = (x[e] * inv) * (float)signs_s[E * lane + e];
  warp_wht<D>(x, lane);
  return n;
}

template <int D, int KIND>
__global__ void __launch_bounds__(kEncThreads) encode_kernel(EncArgs a) {
  using Sh = EncShape<D>;
  constexpr int E = Sh::E;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;

  extern __shared__ __align__(16) unsigned char smem[];
  int8_t* signs_s = reinterpret_cast<int8_t*>(smem);                    // [D]
  float* cb_s = reinterpret_cast<float*>(smem + 256);                  // centroids [8]
  float* bd_s = cb_s + 8;                                              // boundaries [7]
  unsigned char* dyn = smem + 512;

  const DevView& V = a.view;
  const int b = V.idx_bits;
  for (int i = threadIdx.x; i < D; i += blockDim.x) signs_s[i] = a.tab.signs[i];
  if (KIND == kTurboK || KIND == kTurboV) {
    if (threadIdx.x < 8) cb_s[threadIdx.x] = a.tab.centroids[(b - 1) * 8 + threadIdx.x];
    if (threadIdx.x < 7) bd_s[threadIdx.x] = a.tab.boundaries[(b - 1) * 7 + threadIdx.x];
  }
  __syncthreads();
  const int nb = (1 << b) - 1;

  if constexpr (KIND == kTurboK) {
    constexpr int NV = Sh::NV;
    float* r_s = reinterpret_cast<float*>(dyn);                            // [NV][D]
    uint8_t* codes_s = dyn + NV * D * 4;                                   // [NV][D]
    long long* vid_s = reinterpret_cast<long long*>(codes_s + NV * D);     // [NV]
    const long long n_batches = (a.n_vectors + NV - 1) / NV;
    for (long long bt = blockIdx.x; bt < n_batches; bt += gridDim.x) {
      const long long base = bt * NV;
      // ---- phase A: stage 1 and the residual, one warp per vector ----
      for (int v = warp; v < NV; v += kEncWarps) {
        const long long gv = base + v;
        float x[E];
        long long vid = -1;
        if (gv < a.n_vectors) {
          const __half* src;
          vid = enc_locate(a, gv, &src);
          load_vec<D>(src, x, lane);
        } else {
#pragma unroll
          for (int e = 0; e < E; ++e) x[e] = 0.f;
        }
        const float n = stage1_rotate<D>(x, signs_s, lane);
        float rr = 0.f;
#pragma unroll
        for (int e = 0; e < E; ++e) {
          int idx = 0;
          for (int k = 0; k < nb; ++k) idx += (x[e] >= bd_s[k]) ? 1 : 0;
          const float r = x[e] - cb_s[idx];
          rr = fmaf(r, r, rr);
          r_s[v * D + E * lane + e] = r;
          codes_s[v * D + E * lane + e] = (uint8_t)idx;
        }
        const float rnorm = n * sqrtf(warp_sum(rr));
        if (lane == 0) {
          vid_s[v] = vid;
          if (vid >= 0) {
            __half2 hd = __halves2half2(__float2half_rn(n), __float2half_rn(rnorm));
            *reinterpret_cast<__half2*>(V.header + vid * V.hdr_bytes) = hd;
          }
        }
      }
      __syncthreads();
      // ---- phase B: sigma_j = [(S r)_j > 0] for the batch ----
      {
        const int tj = threadIdx.x % Sh::JG, tv = threadIdx.x / Sh::JG;
        float acc[kVPT][4];
#pragma unroll
        for (int v = 0; v < kVPT; ++v)
#pragma unroll
          for (int j = 0; j < 4; ++j) acc[v][j] = 0.f;
        const float* st = a.tab.S_T + 4 * tj;
        const float* rb = r_s + (kVPT * tv) * D;
#pragma unroll 2
        for (int i4 = 0; i4 < D / 4; ++i4) {
          float4 s4[4];
#pragma unroll
          for (int k = 0; k < 4; ++k) s4[k] = __ldg(reinterpret_cast<const float4*>(st + (4 * i4 + k) * D));
#pragma unroll
          for (int v = 0; v < kVPT; ++v) {
            const float4 r4 = *reinterpret_cast<const float4*>(rb + v * D + 4 * i4);
            acc[v][0] = fmaf(r4.x, s4[0].x, acc[v][0]); acc[v][1] = fmaf(r4.x, s4[0].y, acc[v][1]);
            acc[v][2] = fmaf(r4.x, s4[0].z, acc[v][2]); acc[v][3] = fmaf(r4.x, s4[0].w, acc[v][3]);
            acc[v][0] = fmaf(r4.y, s4[1].x, acc[v][0]); acc[v][1] = fmaf(r4.y, s4[1].y, acc[v][1]);
            acc[v][2] = fmaf(r4.y, s4[1].z, acc[v][2]); acc[v][3] = fmaf(r4.y, s4[1].w, acc[v][3]);
            acc[v][0] = fmaf(r4.z, s4[2].x, acc[v][0]); acc[v][1] = fmaf(r4.z, s4[2].y, acc[v][1]);
            acc[v][2] = fmaf(r4.z, s4[2].z, acc[v][2]); acc[v][3] = fmaf(r4.z, s4[2].w, acc[v][3]);
            acc[v][0] = fmaf(r4.w, s4[3].x, acc[v][0]); acc[v][1] = fmaf(r4.w, s4[3].y, acc[v][1]);
            acc[v][2] = fmaf(r4.w, s4[3].z, acc[v][2]); acc[v][3] = fmaf(r4.w, s4[3].w, acc[v][3]);
          }
        }
        const uint8_t sbit = (uint8_t)(1u << b);
#pragma unroll
        for (int v = 0; v < kVPT; ++v)
#pragma unroll
          for (int j = 0; j < 4; ++j)
            if (acc[v][j] > 0.f) codes_s[(kVPT * tv + v) * D + 4 * tj + j] |= sbit;
      }
      __syncthreads();
      // ---- phase C: pack and store ----
      for (int v = warp; v < NV; v += kEncWarps) {
        const long long vid = vid_s[v];
        if (vid >= 0)
          warp_pack_store<D>(codes_s + v * D, V.code_bits,
                             reinterpret_cast<uint32_t*>(V.payload + vid * V.pay_bytes), lane);
      }
      __syncthreads();
    }
  } else {
    uint8_t* codes_s = dyn + warp * D;  // [warps][D]
    const long long gw = (long long)blockIdx.x * kEncWarps + warp;
    const long long nw = (long long)gridDim.x * kEncWarps;
    for (long long gv = gw; gv < a.n_vectors; gv += nw) {
      const __half* src;
      const long long vid = enc_locate(a, gv, &src);
      if (vid < 0) continue;  // warp-uniform
      float x[E];
      load_vec<D>(src, x, lane);
      unsigned char* pay = V.payload + vid * V.pay_bytes;
      unsigned char* hdr = V.header + vid * V.hdr_bytes;
      if constexpr (KIND == kTurboV) {
        const float n = stage1_rotate<D>(x, signs_s, lane);
#pragma unroll
        for (int e = 0; e < E; ++e) {
          int idx = 0;
          for (int k = 0; k < nb; ++k) idx += (x[e] >= bd_s[k]) ? 1 : 0;
          codes_s[E * lane + e] = (uint8_t)idx;
        }
        if (lane == 0) *reinterpret_cast<__half*>(hdr) = __float2half_rn(n);
        __syncwarp();
        warp_pack_store<D>(codes_s, V.code_bits, reinterpret_cast<uint32_t*>(pay), lane);
      } else if constexpr (KIND == kQ8) {
        // block of 32 coordinates = 32/E consecutive lanes
        float amax = 0.f;
#pragma unroll
        for (int e = 0; e < E; ++e) amax = fmaxf(amax, fabsf(x[e]));
#pragma unroll
        for (int m = 1; m < 32 / E; m <<= 1) amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, m));
        const float delta = __fdiv_rn(amax, 127.0f);
        uint32_t packed[E / 2 > 0 ? E / 2 : 1] = {};
#pragma unroll
        for (int e = 0; e < E; ++e) {
          const float qf = delta > 0.f ? roundf(__fdiv_rn(x[e], delta)) : 0.f;
          const uint32_t qb = (uint32_t)(uint8_t)(int8_t)(int)qf;
          packed[e / 4] |= qb << (8 * (e % 4));
        }
        if constexpr (E == 2) {
          reinterpret_cast<uint16_t*>(pay)[lane] = (uint16_t)packed[0];
        } else if constexpr (E == 4) {
          reinterpret_cast<uint32_t*>(pay)[lane] = packed[0];
        } else {
          reinterpret_cast<uint2*>(pay)[lane] = make_uint2(packed[0], packed[1]);
        }
        if ((lane % (32 / E)) == 0)
          reinterpret_cast<__half*>(hdr)[lane / (32 / E)] = __float2half_rn(delta);
      } else {  // kMinMax: groups of 64 coordinates = 64/E consecutive lanes
        float mn = x[0], mx = x[0];
#pragma unroll
        for (int e = 1; e < E; ++e) { mn = fminf(mn, x[e]); mx = fmaxf(mx, x[e]); }
#pragma unroll
        for (int m = 1; m < 64 / E; m <<= 1) {
          mn = fminf(mn, __shfl_xor_sync(kFull, mn, m));
          mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, m));
        }
        const int qmax = (1 << b) - 1;
        const float scale = __fdiv_rn(__fsub_rn(mx, mn), (float)qmax);
#pragma unroll
        for (int e = 0; e < E; ++e) {
          int q = 0;
          if (scale > 0.f) {
            const float t = __fadd_rn(__fdiv_rn(__fsub_rn(x[e], mn), scale), 0.5f);
            q = (int)floorf(t);
            q = q < 0 ? 0 : (q > qmax ? qmax : q);
          }
          codes_s[E * lane + e] = (uint8_t)q;
        }
        if ((lane % (64 / E)) == 0)
          reinterpret_cast<__half2*>(hdr)[lane / (64 / E)] =
              __halves2half2(__float2half_rn(scale), __float2half_rn(mn));
        __syncwarp();
        warp_pack_store<D>(codes_s, V.code_bits, reinterpret_cast<uint32_t*>(pay), lane);
      }
      __syncwarp();
    }
  }
}

template <int D, int KIND>
cudaError_t launch_kind(const EncArgs& a, int sm_count, cudaStream_t s) {
  size_t smem = 512;
  long long work;
  if (KIND == kTurboK) {
    constexpr int NV = EncShape<D>::NV;
    smem += (size_t)NV * D * 5 + NV * 8;
    work = (a.n_vectors + NV - 1) / NV;
  } else {
    smem += (size_t)kEncWarps * D;
    work = (a.n_vectors + kEncWarps - 1) / kEncWarps;
  }
  auto kern = encode_kernel<D, KIND>;
  if (smem > 48 * 1024) {
    const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  int per_sm = 0;
  cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kEncThreads, smem);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) per_sm = 1;
  const long long grid = work < (long long)per_sm * sm_count ? work : (long long)per_sm * sm_count;
  kern<<<(unsigned)grid, kEncThreads, smem, s>>>(a);
  return cudaGetLastError();
}

template <int D>
cudaError_t launch_dim(const EncArgs& a, int sm_count, cudaStream_t s) {
  const int f = a.view.format;
  if (f == TQ_FMT_Q8_0) return launch_kind<D, kQ8>(a, sm_count, s);
  if (f == TQ_FMT_MINMAX) return launch_kind<D, kMinMax>(a, sm_count, s);
  if (a.view.has_qjl) return launch_kind<D, kTurboK>(a, sm_count, s);
  return launch_kind<D, kTurboV>(a, sm_count, s);
}

}  // namespace

cudaError_t launch_encode(const DevTables& t, const DevView& view, const __half* x, int layer_begin,
                          int n_layers, int n_tokens, long long layer_stride, long long token_stride,
                          const long long* slots, long long slot_begin, int sm_count, cudaStream_t s) {
  EncArgs a;
  a.view = view;
  a.tab = t;
  a.x = x;
  a.layer_begin = layer_begin;
  a.n_layers = n_layers;
  a.n_tokens = n_tokens;
  a.layer_stride = layer_stride;
  a.token_stride = token_stride;
  a.slots = slots;
  a.slot_begin = slot_begin;
  a.n_vectors = (long long)n_layers * n_tokens * view.H;
  switch (view.d) {
    case 64: return launch_dim<64>(a, sm_count, s);
    case 128: return launch_dim<128>(a, sm_count, s);
    case 256: return launch_dim<256>(a, sm_count, s);
  }
  return cudaErrorInvalidValue;
}

}  // namespace tq
