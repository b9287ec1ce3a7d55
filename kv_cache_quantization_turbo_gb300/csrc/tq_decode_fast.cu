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
//   * O^T[128 dims x 8 cols] += V~^T . P' on mma.sync m16n8k16 (f16 in, f32
//     accumulate), where P' folds the V norm into the weights.  A 64-entry
//     table indexed by the 6-bit code of two coordinates of one token returns
//     their f16 pair; one prmt per register then pairs two tokens at the same
//     coordinate, which is the fragment layout of a contraction over tokens.
// With up to 4 heads per KV head the 8 mma columns hold each head twice
// (hi and lo fp16 parts of q' and of P'), so the operands keep about 21
// significant bits.
//
// The fp16 tables hold lambda * centroid, lambda chosen on the host so that
// every entry is within ~2e-5 of its fp32 value; 1/lambda goes into the
// per-token norm.
//
// Work: a work item is (layer x sequence, KV head, split of the context); each
// warp takes items from an atomic counter (zeroed by the prologue kernel) and
// writes one partial per query head and item, so warps never wait for each
// other.  Before working on a tile a warp issues that tile's V loads and the
// next tile's K loads.  The running maximum is raised lazily: only when some
// score exceeds it by 2^8 are the sums and accumulators rescaled.
// Two persistent CTAs of 8 warps per SM share the tables of their CTA.
#include <cuda_fp16.h>

#include "tq_device.cuh"

namespace tq {
namespace {

constexpr int kFD = 128;
constexpr int kFWarps = 8;           // warps per CTA; two CTAs per SM
constexpr int kFThreads = kFWarps * 32;

// dynamic shared memory layout (bytes)
constexpr int kLutK = 0;                       // 256 entries x 32 lanes x 8 B
constexpr int kLutV = kLutK + 256 * 256;       // 64 entries x 32 lanes x 4 B
constexpr int kPs = kLutV + 64 * 128;          // per warp P' tile [8 cols][16 tokens] f16
constexpr int kFSmem = kPs + kFWarps * 16 * 8 * 2;

constexpr float kLog2e = 1.4426950408889634074f;
constexpr float kLn2 = 0.6931471805599453094f;
constexpr float kLazyMax = 8.0f;  // rescale only when a score passes the running reference by 2^8

__device__ __forceinline__ uint32_t h2_as_u32(__half2 h) { return *reinterpret_cast<uint32_t*>(&h); }
__device__ __forceinline__ __half2 u32_as_h2(uint32_t u) { return *reinterpret_cast<__half2*>(&u); }

__device__ __forceinline__ void mma_16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                          uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// 2^x for x <= 8 (the scores never exceed the reference by more); -inf -> 0
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
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

__device__ __forceinline__ uint32_t ld_stream_u16(const void* p) {
  unsigned short v;
  asm volatile("ld.global.nc.L1::no_allocate.u16 %0, [%1];" : "=h"(v) : "l"(p));
  return v;
}

// Byte offset of the K table entry for byte kk of word x: (x.byte[kk] << 8) | lane8.
template <int KK>
__device__ __forceinline__ uint32_t lutk_off(uint32_t x, uint32_t lane8) {
  return __byte_perm(x, lane8, 0x7604 | (KK << 4));
}

// Byte offset of the V table entry for the 6-bit code at bit S of w: (code << 7) | lane4.
template <int S>
__device__ __forceinline__ uint32_t lutv_off(uint32_t w, uint32_t lane4) {
  const uint32_t x = S >= 7 ? (w >> (S - 7)) : (w << (7 - S));
  return (x & 0x1F80u) | lane4;
}

// Two f16 B-fragment halves: hi (or lo) part of x0, x1.
__device__ __forceinline__ uint32_t pack_part(float x0, float x1, bool lo) {
  const __half h0 = __float2half_rn(x0), h1 = __float2half_rn(x1);
  if (!lo) return h2_as_u32(__halves2half2(h0, h1));
  return h2_as_u32(__halves2half2(__float2half_rn(x0 - __half2float(h0)), __float2half_rn(x1 - __half2float(h1))));
}

struct KTile {
  uint4 a, b;       // payload blocks of tokens g, g + 8
  uint32_t ha, hb;  // headers (fp16 n, fp16 rnorm)
};
struct VTile {
  uint32_t w[4][2];  // code words of tokens 2t, 2t + 1, 2t + 8, 2t + 9
  uint32_t nv;       // fp16 norms of tokens g (low) and g + 8 (high)
};

// Full tile starting at vector index base: every row is a real token.  Thread
// (g, t) reads K payload block t of tokens g and g + 8, the K headers of g and
// g + 8, V code words vwofs and vwofs + 1 of tokens 2t, 2t + 1, 2t + 8, 2t + 9,
// and the V norms of g and g + 8.
__device__ __forceinline__ void load_k_full(KTile& K, const DecodeArgs& a, long long base, int g, int t) {
  const unsigned char* kp = a.k.payload + (base + g) * 64 + 16 * t;
  const unsigned char* kh = a.k.header + (base + g) * 4;
  K.a = ld_stream_v4(kp);
  K.b = ld_stream_v4(kp + 8 * 64);
  K.ha = ld_stream_u32(kh);
  K.hb = ld_stream_u32(kh + 8 * 4);
}
__device__ __forceinline__ void load_v_full(VTile& V, const DecodeArgs& a, long long base, int g, int t,
                                            int vwofs) {
  const unsigned char* vp = a.v.payload + (base + 2 * t) * 48 + 4 * vwofs;
  const unsigned char* vh = a.v.header + (base + g) * 2;
  const int off[4] = {0, 48, 8 * 48, 9 * 48};
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    V.w[r][0] = ld_stream_u32(vp + off[r]);
    V.w[r][1] = ld_stream_u32(vp + off[r] + 4);
  }
  V.nv = ld_stream_u16(vh) | (ld_stream_u16(vh + 8 * 2) << 16);
}
// Ragged last tile: rows at or beyond nvalid re-read row nvalid - 1 (their scores are masked).
__device__ __forceinline__ void load_k_ragged(KTile& K, const DecodeArgs& a, long long base, int nvalid, int g,
                                              int t) {
  const long long ra = base + min(g, nvalid - 1), rb = base + min(g + 8, nvalid - 1);
  K.a = ld_stream_v4(a.k.payload + ra * 64 + 16 * t);
  K.b = ld_stream_v4(a.k.payload + rb * 64 + 16 * t);
  K.ha = ld_stream_u32(a.k.header + ra * 4);
  K.hb = ld_stream_u32(a.k.header + rb * 4);
}
__device__ __forceinline__ void load_v_ragged(VTile& V, const DecodeArgs& a, long long base, int nvalid, int g,
                                              int t, int vwofs) {
  const int rows[4] = {2 * t, 2 * t + 1, 2 * t + 8, 2 * t + 9};
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    const unsigned char* p = a.v.payload + (base + min(rows[r], nvalid - 1)) * 48 + 4 * vwofs;
    V.w[r][0] = ld_stream_u32(p);
    V.w[r][1] = ld_stream_u32(p + 4);
  }
  V.nv = ld_stream_u16(a.v.header + (base + min(g, nvalid - 1)) * 2) |
         (ld_stream_u16(a.v.header + (base + min(g + 8, nvalid - 1)) * 2) << 16);
}

// Walks the tiles of one work item page by page.  Tiles never straddle pages:
// page_size is a multiple of 16 for paged caches, and a contiguous cache is one page.
struct TileWalk {
  long long base;  // vector index of the current tile's first token
  int in_page;     // token offset of the current tile inside its page
  int page_ord;    // logical page of the sequence
  bool ok;         // current page in range
};

__device__ __forceinline__ long long page_base(const DecodeArgs& a, long long page, int layer, int kvh) {
  return (((long long)layer * a.k.num_pages + page) * a.k.H + kvh) * a.k.page_size;
}

__device__ __forceinline__ void walk_page(TileWalk& W, const DecodeArgs& a, const DecodeLaunch& k, int layer,
                                          int b, int kvh) {
  long long page = b;
  W.ok = true;
  if (a.block_table) {
    page = a.block_table[(long long)b * a.max_blocks_per_seq + W.page_ord];
    if (page < 0 || page >= a.k.num_pages) {
      if ((threadIdx.x & 31) == 0) atomicOr(k.tab.status, kFlagBlockTable);
      W.ok = false;
      page = 0;
    }
  }
  W.base = page_base(a, page, layer, kvh) + W.in_page;
}

template <bool HILO>
__global__ void __launch_bounds__(kFThreads, 2) attend_fast_kernel(DecodeLaunch k) {
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

  const int H = a.k.H, G = k.G, Hq = a.n_q_heads, P = a.k.page_size;
  const unsigned int n_items = (unsigned int)((long long)a.n_layers * a.batch * H * k.n_splits);
  const uint32_t lane8 = (uint32_t)lane << 3, lane4 = (uint32_t)lane << 2;
  __half* Ps = reinterpret_cast<__half*>(sm + kPs) + warp * 128;  // P' as [8 cols][16 tokens] fp16
  const float kq = kSqrtHalfPi / (float)kFD;
  const float inv_lam = 1.0f / k.tab.f16_scale[2];
  const float tau = a.skip_threshold;
  // V codes of coordinates [16g, 16g + 16) sit at bits [48g, 48g + 48) of the payload
  const int vwofs = (3 * g) >> 1, vsh = (g & 1) ? 16 : 0;

  for (;;) {
    unsigned int item = 0;
    if (lane == 0) item = atomicAdd(k.counter, 1u);
    item = __shfl_sync(kFull, item, 0);
    if (item >= n_items) break;
    const int split = (int)(item % k.n_splits);
    const unsigned int rest = item / k.n_splits;
    const int kvh = (int)(rest % H);
    const int lb = (int)(rest / H);
    const int layer = a.layer_begin + lb / a.batch, b = lb % a.batch;
    int len = a.seq_lens[b];
    if (len < 0) len = 0;
    if (len > a.max_ctx) {
      if (lane == 0) atomicOr(k.tab.status, kFlagSeqLen);
      len = a.max_ctx;
    }
    const int t0 = split * k.split_tokens;
    const int t1 = min(t0 + k.split_tokens, len);
    const long long row0 = (long long)lb * Hq + (long long)kvh * G;

    // ---- B fragments of q' (chain 1) and S q' (chain 2), column g; log2 e folded in ----
    uint32_t bq[8][2], bs[8][2];
    {
      const int head = HILO ? (g & 3) : g;
      const bool lo_part = HILO && g >= 4;
      const bool valid = head < G;
      const float* qp = k.qprep + (row0 + (valid ? head : 0)) * 2 * kFD + 32 * t;
      const float f = valid ? kLog2e : 0.f;
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        const float4 qv = *reinterpret_cast<const float4*>(qp + 4 * c);
        const float4 sv = *reinterpret_cast<const float4*>(qp + kFD + 4 * c);
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
    TileWalk Wk;
    KTile kc, kn;
    VTile vc;
    if (ntiles > 0) {
      Wk.page_ord = t0 / P;
      Wk.in_page = t0 - Wk.page_ord * P;
      walk_page(Wk, a, k, layer, b, kvh);
      if (ntiles == 1 && t1 - t0 < 16) load_k_ragged(kc, a, Wk.base, t1 - t0, g, t);
      else load_k_full(kc, a, Wk.base, g, t);
    }
    for (int tile = 0; tile < ntiles; ++tile) {
      const int nvalid = min(16, t1 - (t0 + 16 * tile));
      const bool cur_ok = Wk.ok;
      const long long cur_base = Wk.base;
      if (nvalid == 16) load_v_full(vc, a, cur_base, g, t, vwofs);
      else load_v_ragged(vc, a, cur_base, nvalid, g, t, vwofs);
      // next tile: address and K loads
      if (tile + 1 < ntiles) {
        Wk.in_page += 16;
        if (Wk.in_page == P) {  // next page
          Wk.in_page = 0;
          ++Wk.page_ord;
          walk_page(Wk, a, k, layer, b, kvh);
        } else {
          Wk.base += 16;
        }
        const int nvn = min(16, t1 - (t0 + 16 * (tile + 1)));
        if (nvn == 16) load_k_full(kn, a, Wk.base, g, t);
        else load_k_ragged(kn, a, Wk.base, nvn, g, t);
      }
      do {
        if (!cur_ok) break;  // warp-uniform: the tile's page was out of range
        // ---- K: table dequantisation, two mma chains ----
        float cm[4] = {0.f, 0.f, 0.f, 0.f}, cq[4] = {0.f, 0.f, 0.f, 0.f};
        const uint32_t wa[4] = {kc.a.x, kc.a.y, kc.a.z, kc.a.w};
        const uint32_t wb[4] = {kc.b.x, kc.b.y, kc.b.z, kc.b.w};
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
        // rows g (c0, c1) and g + 8 (c2, c3), columns 2t, 2t + 1; scores in log2 units
        const float2 hA = __half22float2(u32_as_h2(kc.ha)), hB = __half22float2(u32_as_h2(kc.hb));
        const float nA = hA.x * inv_lam, nB = hB.x * inv_lam, rA = hA.y * kq, rB = hB.y * kq;
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
        if (nvalid < 16) {
          if (g >= nvalid) s0 = s1 = -INFINITY;
          if (g + 8 >= nvalid) s2 = s3 = -INFINITY;
        }

        // ---- online softmax with a lazily raised reference (base 2) ----
        {
          float mx0 = fmaxf(s0, s2), mx1 = fmaxf(s1, s3);
          if (__any_sync(kFull, mx0 > m0 + kLazyMax || mx1 > m1 + kLazyMax)) {
#pragma unroll
            for (int o = 4; o < 32; o <<= 1) {
              mx0 = fmaxf(mx0, __shfl_xor_sync(kFull, mx0, o));
              mx1 = fmaxf(mx1, __shfl_xor_sync(kFull, mx1, o));
            }
            const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
            const float al0 = ex2(m0 - mn0), al1 = ex2(m1 - mn1);
            l0 *= al0;
            l1 *= al1;
#pragma unroll
            for (int mt = 0; mt < 8; ++mt) {
              oacc[mt][0] *= al0; oacc[mt][1] *= al1; oacc[mt][2] *= al0; oacc[mt][3] *= al1;
            }
            m0 = mn0;
            m1 = mn1;
          }
        }
        float p0 = ex2(s0 - m0), p1 = ex2(s1 - m1), p2 = ex2(s2 - m0), p3 = ex2(s3 - m1);
        l0 += p0 + p2;
        l1 += p1 + p3;
        // ---- Sparse V: weights below the threshold are dropped; an all-dropped tile skips V ----
        p0 = p0 >= tau ? p0 : 0.f;
        p1 = p1 >= tau ? p1 : 0.f;
        p2 = p2 >= tau ? p2 : 0.f;
        p3 = p3 >= tau ? p3 : 0.f;
        if (!__any_sync(kFull, (p0 + p1 + p2 + p3) > 0.f)) break;

        // ---- P' = p * n_v / lambda as fp16 hi/lo, transposed to [col][token] in shared memory ----
        const float2 nv = __half22float2(u32_as_h2(vc.nv));
        const float nvA = nv.x * inv_lam, nvB = nv.y * inv_lam;
        const float w[4] = {p0 * nvA, p1 * nvA, p2 * nvB, p3 * nvB};
        __half hw[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const __half hi = __float2half_rn(w[i]);
          hw[i] = (HILO && t >= 2) ? __float2half_rn(w[i] - __half2float(hi)) : hi;
        }
        __syncwarp();
        Ps[(2 * t) * 16 + g] = hw[0];
        Ps[(2 * t + 1) * 16 + g] = hw[1];
        Ps[(2 * t) * 16 + g + 8] = hw[2];
        Ps[(2 * t + 1) * 16 + g + 8] = hw[3];
        __syncwarp();
        const uint32_t bp0 = *reinterpret_cast<const uint32_t*>(Ps + g * 16 + 2 * t);
        const uint32_t bp1 = *reinterpret_cast<const uint32_t*>(Ps + g * 16 + 2 * t + 8);

        // ---- V: O^T[16 dims x 8 cols] += V~^T[16 dims x 16 tokens] . P'[16 tokens x 8 cols] ----
        // rows g / g + 8 of m-tile mt = coordinates 16g + 2mt / +1; k-slots = tokens of the tile
        uint32_t xl[4], xh[4];
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          xl[r] = __funnelshift_r(vc.w[r][0], vc.w[r][1], vsh);
          xh[r] = vc.w[r][1] >> vsh;
        }
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) {
          uint32_t e[4];
#pragma unroll
          for (int r = 0; r < 4; ++r) {
            uint32_t o;
            switch (mt) {
              case 0: o = lutv_off<0>(xl[r], lane4); break;
              case 1: o = lutv_off<6>(xl[r], lane4); break;
              case 2: o = lutv_off<12>(xl[r], lane4); break;
              case 3: o = lutv_off<18>(xl[r], lane4); break;
              case 4: o = lutv_off<24>(xl[r], lane4); break;
              case 5: o = lutv_off<7>(__funnelshift_r(xl[r], xh[r], 23), lane4); break;
              case 6: o = lutv_off<4>(xh[r], lane4); break;
              default: o = lutv_off<10>(xh[r], lane4); break;
            }
            e[r] = *reinterpret_cast<const uint32_t*>(sm + kLutV + o);  // (c[2p], c[2p+1]) of one token
          }
          // a0/a1: tokens 2t, 2t+1 at coordinate 2p / 2p+1; a2/a3: tokens 2t+8, 2t+9
          mma_16816(oacc[mt], __byte_perm(e[0], e[1], 0x5410), __byte_perm(e[0], e[1], 0x7632),
                    __byte_perm(e[2], e[3], 0x5410), __byte_perm(e[2], e[3], 0x7632), bp0, bp1);
        }
      } while (0);
      if (tile + 1 < ntiles) kc = kn;
    }

    // ---- partial of this work item: (m, l, acc) per query head ----
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) {
      l0 += __shfl_xor_sync(kFull, l0, o);
      l1 += __shfl_xor_sync(kFull, l1, o);
    }
    if (HILO) {  // add the lo columns (t = 2, 3) into the hi columns (t = 0, 1)
#pragma unroll
      for (int mt = 0; mt < 8; ++mt)
#pragma unroll
        for (int e = 0; e < 4; ++e) oacc[mt][e] += __shfl_xor_sync(kFull, oacc[mt][e], 2);
    }
    const int h0 = HILO ? 2 * (t & 1) : 2 * t;
    const bool writer = !HILO || t < 2;
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int h = h0 + e;
      if (!writer || h >= G) continue;
      float* dst = k.partial + ((row0 + h) * k.n_splits + split) * (kFD + 4);
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) {
        dst[4 + 16 * g + 2 * mt] = oacc[mt][e];
        dst[4 + 16 * g + 2 * mt + 1] = oacc[mt][2 + e];
      }
      if (g == 0) {
        const float m = e ? m1 : m0, l = e ? l1 : l0;
        dst[0] = m == -INFINITY ? -INFINITY : m * kLn2;
        dst[1] = l;
      }
    }
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
  const long long warps = (items + 0);  // one warp per item at most
  long long grid = 2LL * sm_count;
  if (warps < grid * kFWarps) grid = (warps + kFWarps - 1) / kFWarps;
  if (items >= (1LL << 32)) return cudaErrorInvalidValue;
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
