// Split-K decode attention on tensor cores for turbo4 K (3-bit index + QJL
// sign per coordinate, stored as nibbles) and turbo4_mse V (3-bit index),
// head_dim 128, up to 8 query heads per KV head.  Same contract as the
// generic kernel in tq_decode.cu: one partial (m, l, acc) per (query row,
// split), combined afterwards.
//
// Per warp, tiles of 16 tokens:
//   * scores S^T[16 tokens x 8 cols] = K~[16 x 128] . Q^T on mma.sync
//     m16n8k16 (f16 in, f32 accumulate), two chains: the codebook part
//     c[idx] against q' and the QJL part (2 sigma - 1) against S q'.  The A
//     fragments come from a 256-entry table in shared memory indexed by one
//     payload byte (two coordinates: index + sign nibbles) that returns both
//     f16 pairs at once; the table is replicated per lane (entry stride 256 B,
//     lane offset 8 B) so the 32 lookups of a warp never collide, and one
//     prmt forms the address (byte << 8 | lane << 3).
//     score = n * chain1 + rnorm * sqrt(pi/2)/d * chain2 (per token).
//   * online softmax in registers (base-2: log2 e is folded into q'),
//   * Sparse V: a tile whose every weight is below the threshold skips V,
//     inside a kept tile weights below it are zeroed;
//   * O^T[128 dims x 8 cols] += V~^T . P' on mma.sync m16n8k8 tf32, where P'
//     folds the V norm into the weights; V A fragments come from a 64-entry
//     table of f16 pairs indexed by the 6-bit code of two coordinates.
// With up to 4 heads per KV head the 8 mma columns hold each head twice
// (hi and lo fp16 parts of q', hi and lo tf32 parts of P'), so the operands
// keep about 21 significant bits.
//
// The fp16 tables hold lambda * centroid, lambda chosen on the host so that
// every entry is within ~2e-5 of its fp32 value; 1/lambda goes into the
// per-token norm.  Each warp issues all loads of its next tile (K and V codes
// and norms) before working on the current one.
//
// CTA: 12 warps over the 16-token tiles of one work item (layer x sequence,
// KV head, split), merged through shared memory; one persistent CTA per SM.
#include <cuda_fp16.h>

#include "tq_device.cuh"

namespace tq {
namespace {

constexpr int kFD = 128;
constexpr int kFWarps = 12;
constexpr int kFThreads = kFWarps * 32;

// dynamic shared memory layout (bytes)
constexpr int kLutK = 0;                       // 256 entries x 32 lanes x 8 B
constexpr int kLutV = kLutK + 256 * 256;       // 64 entries x 32 lanes x 4 B
constexpr int kPs = kLutV + 64 * 128;          // per warp P' tile [16 tokens][8 cols] f32
constexpr int kMAcc = kPs + kFWarps * 16 * 8 * 4;   // per warp O [8 cols][128 dims] f32
constexpr int kMML = kMAcc + kFWarps * 8 * kFD * 4;  // per warp (m, l) [8 cols][2] f32
constexpr int kFSmem = kMML + kFWarps * 8 * 2 * 4;

constexpr float kLog2e = 1.4426950408889634074f;
constexpr float kLn2 = 0.6931471805599453094f;

__device__ __forceinline__ uint32_t h2_as_u32(__half2 h) { return *reinterpret_cast<uint32_t*>(&h); }
__device__ __forceinline__ __half2 u32_as_h2(uint32_t u) { return *reinterpret_cast<__half2*>(&u); }

__device__ __forceinline__ void mma_16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                          uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void mma_1688_tf32(float (&c)[4], float a0, float a1, float a2, float a3, float b0,
                                              float b1) {
  asm("mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(__float_as_uint(a0)), "r"(__float_as_uint(a1)), "r"(__float_as_uint(a2)), "r"(__float_as_uint(a3)),
        "r"(__float_as_uint(b0)), "r"(__float_as_uint(b1)));
}

__device__ __forceinline__ float tf32_rna(float x) {
  uint32_t r;
  asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
  return __uint_as_float(r);
}

__device__ __forceinline__ uint4 ld_stream_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ uint32_t ld_stream_u32(const void* p) {
  uint32_t v;
  asm volatile("ld.global.nc.L1::no_allocate.u32 %0, [%1];" : "=r"(v) : "l"(p));
  return v;
}

// Byte offset of the K table entry for byte kk of word x: (x.byte[kk] << 8) | lane8.
template <int KK>
__device__ __forceinline__ uint32_t lutk_off(uint32_t x, uint32_t lane8) {
  return __byte_perm(x, lane8, 0x7604 | (KK << 4));
}

// Two f16 B-fragment halves: hi (or lo) part of x0, x1.
__device__ __forceinline__ uint32_t pack_part(float x0, float x1, bool lo) {
  const __half h0 = __float2half_rn(x0), h1 = __float2half_rn(x1);
  if (!lo) return h2_as_u32(__halves2half2(h0, h1));
  return h2_as_u32(__halves2half2(__float2half_rn(x0 - __half2float(h0)), __float2half_rn(x1 - __half2float(h1))));
}

// Everything a warp loads for one 16-token tile, issued one tile ahead.
struct TileIn {
  uint4 kA, kB;          // K payload block t of tokens g and g + 8 (16 B each)
  uint32_t hA, hB;       // K headers (fp16 n, fp16 rnorm) of tokens g and g + 8
  uint32_t nv;           // V norms (fp16) of tokens g and g + 8
  uint32_t v[2][2][2];   // V code words [k-step][token t / t + 4][2 words]
  int nvalid;            // tokens of the tile inside [t0, t1)
  bool ok;               // the tile's page is in range
};

__device__ __forceinline__ void load_tile(TileIn& T, const DecodeArgs& a, const DecodeLaunch& k, int tile, int t0,
                                          int t1, int layer, int b, int kvh, int g, int t, int vwofs) {
  const int j0 = t0 + tile * 16;
  T.nvalid = min(16, t1 - j0);
  long long page = b;
  T.ok = true;
  if (a.block_table) {
    page = a.block_table[(long long)b * a.max_blocks_per_seq + j0 / a.k.page_size];
    if (page < 0 || page >= a.k.num_pages) {
      if ((threadIdx.x & 31) == 0) atomicOr(k.tab.status, kFlagBlockTable);
      T.ok = false;
      return;
    }
  }
  // tiles never cross a page: page_size is a multiple of 16 (or the cache is contiguous)
  const long long base = (((long long)layer * a.k.num_pages + page) * a.k.H + kvh) * a.k.page_size +
                         (j0 % a.k.page_size);
  const int last = T.nvalid - 1;
  const long long rA = base + min(g, last), rB = base + min(g + 8, last);
  T.kA = ld_stream_v4(a.k.payload + rA * 64 + 16 * t);
  T.kB = ld_stream_v4(a.k.payload + rB * 64 + 16 * t);
  T.hA = ld_stream_u32(a.k.header + rA * 4);
  T.hB = ld_stream_u32(a.k.header + rB * 4);
  const uint32_t nva = *reinterpret_cast<const unsigned short*>(a.v.header + rA * 2);
  const uint32_t nvb = *reinterpret_cast<const unsigned short*>(a.v.header + rB * 2);
  T.nv = nva | (nvb << 16);
#pragma unroll
  for (int ks = 0; ks < 2; ++ks) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const long long r = base + min(8 * ks + t + 4 * h, last);
      const unsigned char* p = a.v.payload + r * 48 + 4 * vwofs;
      T.v[ks][h][0] = ld_stream_u32(p);
      T.v[ks][h][1] = ld_stream_u32(p + 4);
    }
  }
}

template <bool HILO>
__global__ void __launch_bounds__(kFThreads, 1) attend_fast_kernel(DecodeLaunch k) {
  extern __shared__ __align__(16) unsigned char sm[];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, t = lane & 3;
  const DecodeArgs& a = k.a;

  // ---- tables (once per persistent CTA) ----
  {
    const float* cb = k.tab.centroids + 2 * 8;  // 3-bit codebook
    const float lam = k.tab.f16_scale[2];
    for (int i = tid; i < 256 * 32; i += kFThreads) {
      const int e = i >> 5, r = i & 31, lo = e & 15, hi = e >> 4;
      uint2 v;
      v.x = h2_as_u32(__floats2half2_rn(lam * cb[lo & 7], lam * cb[hi & 7]));
      v.y = h2_as_u32(__floats2half2_rn((lo >> 3) ? 1.f : -1.f, (hi >> 3) ? 1.f : -1.f));
      *reinterpret_cast<uint2*>(sm + kLutK + e * 256 + r * 8) = v;
    }
    for (int i = tid; i < 64 * 32; i += kFThreads) {
      const int e = i >> 5, r = i & 31;
      *reinterpret_cast<uint32_t*>(sm + kLutV + e * 128 + r * 4) =
          h2_as_u32(__floats2half2_rn(lam * cb[e & 7], lam * cb[e >> 3]));
    }
  }
  __syncthreads();

  const int H = a.k.H, G = k.G, Hq = a.n_q_heads;
  const long long n_items = (long long)a.n_layers * a.batch * H * k.n_splits;
  const uint32_t lane8 = (uint32_t)lane << 3, lane4 = (uint32_t)lane << 2;
  float* Ps = reinterpret_cast<float*>(sm + kPs) + warp * 128;
  const float kq = kSqrtHalfPi / (float)kFD;
  const float tau = a.skip_threshold;
  // V codes of coordinates [16g, 16g + 16) sit at bits [48g, 48g + 48) of the payload
  const int vwofs = (3 * g) >> 1, vsh = (g & 1) ? 16 : 0;

  for (long long item = blockIdx.x; item < n_items; item += gridDim.x) {
    const int split = (int)(item % k.n_splits);
    const long long rest = item / k.n_splits;
    const int kvh = (int)(rest % H);
    const int lb = (int)(rest / H);
    const int layer = a.layer_begin + lb / a.batch, b = lb % a.batch;
    int len = a.seq_lens[b];
    if (len < 0) len = 0;
    if (len > a.max_ctx) {
      if (tid == 0) atomicOr(k.tab.status, kFlagSeqLen);
      len = a.max_ctx;
    }
    const int t0 = split * k.split_tokens;
    const int t1 = min(t0 + k.split_tokens, len);
    const long long row0 = (long long)lb * Hq + (long long)kvh * G;

    // ---- B fragments of q' (chain 1) and S q' (chain 2), column g ----
    uint32_t bq[8][2], bs[8][2];
    {
      const int head = HILO ? (g & 3) : g;
      const bool lo_part = HILO && g >= 4;
      const bool valid = head < G;
      const float* qp = k.qprep + (row0 + (valid ? head : 0)) * 2 * kFD + 32 * t;
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        float4 qv = *reinterpret_cast<const float4*>(qp + 4 * c);
        float4 sv = *reinterpret_cast<const float4*>(qp + kFD + 4 * c);
        const float f = valid ? kLog2e : 0.f;
        bq[c][0] = pack_part(qv.x * f, qv.y * f, lo_part);
        bq[c][1] = pack_part(qv.z * f, qv.w * f, lo_part);
        bs[c][0] = pack_part(sv.x * f, sv.y * f, lo_part);
        bs[c][1] = pack_part(sv.z * f, sv.w * f, lo_part);
      }
    }
    float oacc[8][4];
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) oacc[mt][0] = oacc[mt][1] = oacc[mt][2] = oacc[mt][3] = 0.f;
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;

    const int ntiles = t1 > t0 ? (t1 - t0 + 15) / 16 : 0;
    const float nk_scale = 1.0f / k.tab.f16_scale[2];   // undo lambda of the K table (chain 1)
    TileIn cur, nxt;
    int tile = warp;
    if (tile < ntiles) load_tile(cur, a, k, tile, t0, t1, layer, b, kvh, g, t, vwofs);
    for (; tile < ntiles; tile += kFWarps) {
      if (tile + kFWarps < ntiles) load_tile(nxt, a, k, tile + kFWarps, t0, t1, layer, b, kvh, g, t, vwofs);
      do {
        if (!cur.ok) break;  // warp-uniform: the tile's page was out of range
        const int nvalid = cur.nvalid;
        // ---- K: table dequantisation, two mma chains ----
        float cm[4] = {0.f, 0.f, 0.f, 0.f}, cq[4] = {0.f, 0.f, 0.f, 0.f};
        const uint32_t wa[4] = {cur.kA.x, cur.kA.y, cur.kA.z, cur.kA.w};
        const uint32_t wb[4] = {cur.kB.x, cur.kB.y, cur.kB.z, cur.kB.w};
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const uint32_t xa = wa[c >> 1], xb = wb[c >> 1];
          uint32_t oa0, ob0, oa1, ob1;
          if (c & 1) {
            oa0 = lutk_off<2>(xa, lane8); ob0 = lutk_off<2>(xb, lane8);
            oa1 = lutk_off<3>(xa, lane8); ob1 = lutk_off<3>(xb, lane8);
          } else {
            oa0 = lutk_off<0>(xa, lane8); ob0 = lutk_off<0>(xb, lane8);
            oa1 = lutk_off<1>(xa, lane8); ob1 = lutk_off<1>(xb, lane8);
          }
          const uint2 ea0 = *reinterpret_cast<const uint2*>(sm + kLutK + oa0);
          const uint2 eb0 = *reinterpret_cast<const uint2*>(sm + kLutK + ob0);
          const uint2 ea1 = *reinterpret_cast<const uint2*>(sm + kLutK + oa1);
          const uint2 eb1 = *reinterpret_cast<const uint2*>(sm + kLutK + ob1);
          mma_16816(cm, ea0.x, eb0.x, ea1.x, eb1.x, bq[c][0], bq[c][1]);
          mma_16816(cq, ea0.y, eb0.y, ea1.y, eb1.y, bs[c][0], bs[c][1]);
        }
        // rows g (c0, c1) and g + 8 (c2, c3), columns 2t, 2t + 1
        const float2 hA = __half22float2(u32_as_h2(cur.hA)), hB = __half22float2(u32_as_h2(cur.hB));
        const float nA = hA.x * nk_scale, nB = hB.x * nk_scale, rA = hA.y * kq, rB = hB.y * kq;
        float s0 = fmaf(nA, cm[0], rA * cq[0]);
        float s1 = fmaf(nA, cm[1], rA * cq[1]);
        float s2 = fmaf(nB, cm[2], rB * cq[2]);
        float s3 = fmaf(nB, cm[3], rB * cq[3]);
        if (HILO) {
          s0 += __shfl_xor_sync(kFull, s0, 2);
          s1 += __shfl_xor_sync(kFull, s1, 2);
          s2 += __shfl_xor_sync(kFull, s2, 2);
          s3 += __shfl_xor_sync(kFull, s3, 2);
        }
        if (g >= nvalid) s0 = s1 = -INFINITY;
        if (g + 8 >= nvalid) s2 = s3 = -INFINITY;

        // ---- online softmax (base 2) ----
        float mx0 = fmaxf(s0, s2), mx1 = fmaxf(s1, s3);
#pragma unroll
        for (int o = 4; o < 32; o <<= 1) {
          mx0 = fmaxf(mx0, __shfl_xor_sync(kFull, mx0, o));
          mx1 = fmaxf(mx1, __shfl_xor_sync(kFull, mx1, o));
        }
        const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
        const float al0 = exp2f(m0 - mn0), al1 = exp2f(m1 - mn1);
        float p0 = exp2f(s0 - mn0), p1 = exp2f(s1 - mn1), p2 = exp2f(s2 - mn0), p3 = exp2f(s3 - mn1);
        l0 = fmaf(l0, al0, p0 + p2);
        l1 = fmaf(l1, al1, p1 + p3);
        m0 = mn0;
        m1 = mn1;
        if (__any_sync(kFull, al0 != 1.f || al1 != 1.f)) {
#pragma unroll
          for (int mt = 0; mt < 8; ++mt) {
            oacc[mt][0] *= al0; oacc[mt][1] *= al1; oacc[mt][2] *= al0; oacc[mt][3] *= al1;
          }
        }
        // ---- Sparse V ----
        p0 = p0 >= tau ? p0 : 0.f;
        p1 = p1 >= tau ? p1 : 0.f;
        p2 = p2 >= tau ? p2 : 0.f;
        p3 = p3 >= tau ? p3 : 0.f;
        if (!__any_sync(kFull, (p0 + p1 + p2 + p3) > 0.f)) break;

        // ---- P' = p * n_v / lambda (tf32 hi/lo), transposed through shared memory ----
        const float2 nv = __half22float2(u32_as_h2(cur.nv));
        const float nvA = nv.x * nk_scale, nvB = nv.y * nk_scale;
        float w0 = p0 * nvA, w1 = p1 * nvA, w2 = p2 * nvB, w3 = p3 * nvB;
        if (HILO) {
          const bool lo = t >= 2;
          const float h0 = tf32_rna(w0), h1 = tf32_rna(w1), h2 = tf32_rna(w2), h3 = tf32_rna(w3);
          w0 = lo ? w0 - h0 : h0; w1 = lo ? w1 - h1 : h1; w2 = lo ? w2 - h2 : h2; w3 = lo ? w3 - h3 : h3;
        } else {
          w0 = tf32_rna(w0); w1 = tf32_rna(w1); w2 = tf32_rna(w2); w3 = tf32_rna(w3);
        }
        __syncwarp();
        *reinterpret_cast<float2*>(Ps + g * 8 + 2 * t) = make_float2(w0, w1);
        *reinterpret_cast<float2*>(Ps + (g + 8) * 8 + 2 * t) = make_float2(w2, w3);
        __syncwarp();
        const float bp[4] = {Ps[t * 8 + g], Ps[(t + 4) * 8 + g], Ps[(8 + t) * 8 + g], Ps[(12 + t) * 8 + g]};

        // ---- V: table dequantisation, mma ----
#pragma unroll
        for (int ks = 0; ks < 2; ++ks) {
          const unsigned long long xa =
              (((unsigned long long)cur.v[ks][0][1] << 32) | cur.v[ks][0][0]) >> vsh;
          const unsigned long long xb =
              (((unsigned long long)cur.v[ks][1][1] << 32) | cur.v[ks][1][0]) >> vsh;
#pragma unroll
          for (int mt = 0; mt < 8; ++mt) {
            const uint32_t oa = (((uint32_t)(xa >> (6 * mt)) & 63u) << 7) | lane4;
            const uint32_t ob = (((uint32_t)(xb >> (6 * mt)) & 63u) << 7) | lane4;
            const float2 fa = __half22float2(u32_as_h2(*reinterpret_cast<const uint32_t*>(sm + kLutV + oa)));
            const float2 fb = __half22float2(u32_as_h2(*reinterpret_cast<const uint32_t*>(sm + kLutV + ob)));
            // rows g / g + 8 = coordinates 16g + 2mt / +1; columns t / t + 4 = tokens 8ks + t / + 4
            mma_1688_tf32(oacc[mt], fa.x, fa.y, fb.x, fb.y, bp[2 * ks], bp[2 * ks + 1]);
          }
        }
      } while (0);
      cur = nxt;
    }

    // ---- merge the warps and write the partial of every query head ----
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) {
      l0 += __shfl_xor_sync(kFull, l0, o);
      l1 += __shfl_xor_sync(kFull, l1, o);
    }
    float* macc = reinterpret_cast<float*>(sm + kMAcc) + warp * 8 * kFD;
    float* mml = reinterpret_cast<float*>(sm + kMML) + warp * 16;
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) {
      const int d0 = 16 * g + 2 * mt;
      macc[(2 * t) * kFD + d0] = oacc[mt][0];
      macc[(2 * t + 1) * kFD + d0] = oacc[mt][1];
      macc[(2 * t) * kFD + d0 + 1] = oacc[mt][2];
      macc[(2 * t + 1) * kFD + d0 + 1] = oacc[mt][3];
    }
    if (g == 0) {
      mml[(2 * t) * 2] = m0; mml[(2 * t) * 2 + 1] = l0;
      mml[(2 * t + 1) * 2] = m1; mml[(2 * t + 1) * 2 + 1] = l1;
    }
    __syncthreads();
    const float* macc_all = reinterpret_cast<const float*>(sm + kMAcc);
    const float* mml_all = reinterpret_cast<const float*>(sm + kMML);
    for (int o = tid; o < G * kFD; o += kFThreads) {
      const int h = o / kFD, i = o % kFD;
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < kFWarps; ++w) M = fmaxf(M, mml_all[w * 16 + h * 2]);
      float L = 0.f, acc = 0.f;
      if (M != -INFINITY) {
#pragma unroll
        for (int w = 0; w < kFWarps; ++w) {
          const float mw = mml_all[w * 16 + h * 2];
          if (mw == -INFINITY) continue;
          const float f = exp2f(mw - M);
          L = fmaf(mml_all[w * 16 + h * 2 + 1], f, L);
          float v = macc_all[(w * 8 + h) * kFD + i];
          if (HILO) v += macc_all[(w * 8 + h + 4) * kFD + i];
          acc = fmaf(v, f, acc);
        }
      }
      float* dst = k.partial + ((row0 + h) * k.n_splits + split) * (kFD + 4);
      dst[4 + i] = acc;
      if (i == 0) {
        dst[0] = M == -INFINITY ? -INFINITY : M * kLn2;
        dst[1] = L;
      }
    }
    __syncthreads();
  }
}

}  // namespace

bool attend_fast_supported(const DecodeLaunch& k) {
  const DecodeArgs& a = k.a;
  return a.k.d == kFD && a.k.format == TQ_FMT_TURBO4 && a.v.format == TQ_FMT_TURBO4_MSE && k.G >= 1 &&
         k.G <= 8 && (a.block_table == nullptr || a.k.page_size % 16 == 0) && k.split_tokens % 16 == 0;
}

cudaError_t launch_attend_fast(const DecodeLaunch& k, int sm_count, cudaStream_t s) {
  const long long items = (long long)k.a.n_layers * k.a.batch * k.a.k.H * k.n_splits;
  const long long grid = items < (long long)sm_count ? items : (long long)sm_count;
  if (k.G <= 4) {
    cudaError_t e = cudaFuncSetAttribute(attend_fast_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, kFSmem);
    if (e != cudaSuccess) return e;
    attend_fast_kernel<true><<<(unsigned)grid, kFThreads, kFSmem, s>>>(k);
  } else {
    cudaError_t e = cudaFuncSetAttribute(attend_fast_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, kFSmem);
    if (e != cudaSuccess) return e;
    attend_fast_kernel<false><<<(unsigned)grid, kFThreads, kFSmem, s>>>(k);
  }
  return cudaGetLastError();
}

}  // namespace tq
