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
//     the E = d/32 consecutive coordinates [E l, E l + E); the sign flips, the
//     codebook boundaries and the WHT butterfly signs live in registers;
//   - the Lloyd-Max index is a binary search over the sorted boundaries (the
//     count of boundaries <= y, ties included as the definition has it);
//   - codes are packed by warp shuffles: lane l forms the E w-bit codes of its
//     coordinates as one chunk, and lane j gathers the chunks that overlap
//     32-bit word j of the little-endian stream;
//   - turbo K: a CTA encodes a batch of NV = 8192/d vectors: phase A (warps:
//     stage 1, the residual r into shared memory), phase B (the whole CTA: the
//     d x d projection S r on mma.sync m16n8k16, f16 inputs split into high and
//     low parts, r_hi s_hi + r_lo s_hi + r_hi s_lo accumulated in fp32, which
//     leaves an error near 1e-7 of |r|, far inside the 1e-6 sign band), phase C
//     (warps: pack codes and store);
//   - vector ids -> (layer, token, head) and slots -> (page, offset) use
//     multiply-shift division by invariant divisors;
//   - grids are persistent: min(work, resident CTAs) CTAs loop over batches.
#include <cuda_fp16.h>

#include "tq_device.cuh"

namespace tq {
namespace {

enum EncKind { kTurboK = 0, kTurboV = 1, kQ8 = 2, kMinMax = 3 };

constexpr int kEncThreads = 256;
constexpr int kEncWarps = kEncThreads / 32;
constexpr float kRScale = 16384.0f;  // residual scale before the fp16 split (only signs are kept)

// Unsigned division by an invariant divisor (Granlund-Montgomery, round-up multiplier).
struct FastDiv {
  uint32_t d, m;
  uint32_t s1, s2;
};

FastDiv make_fastdiv(uint32_t d) {
  if (d == 0) d = 1;  // never used with 0 (empty calls return before launching)
  int l = 0;
  while ((1ull << l) < d) ++l;
  const uint64_t m = ((1ull << 32) * ((1ull << l) - d)) / d + 1;
  return FastDiv{d, (uint32_t)m, l ? 1u : 0u, l ? (uint32_t)(l - 1) : 0u};
}

__device__ __forceinline__ uint32_t fdiv(uint32_t n, const FastDiv& f) {
  const uint32_t t = __umulhi(n, f.m);
  return (t + ((n - t) >> f.s1)) >> f.s2;
}

template <int D>
struct EncShape {
  static constexpr int E = D / 32;
  static constexpr int NV = 8192 / D;   // vectors per batch (turbo K)
  static constexpr int RS = D + 8;      // row stride of the residual tile (floats)
  static constexpr int KS = D / 16;     // k steps of the projection
};

struct EncArgs {
  DevView view;
  DevTables tab;
  const __half* x;
  int layer_begin, n_layers, n_tokens;
  long long layer_stride, token_stride;
  const long long* slots;
  long long slot_begin;
  long long n_vectors;  // n_layers * n_tokens * H (< 2^32)
  FastDiv div_h, div_t, div_p;
  int slot32;           // slot capacity below 2^32: the page division is 32-bit
};

// Location of one vector: input address and destination index (-1: skipped).
struct Loc {
  const __half* src;
  long long vid;
};

// The H vectors of a token share everything but the head: the token's input address and
// destination (head 0) are kept and reused while consecutive vectors stay in that token.
struct TokenCache {
  uint32_t lt = 0xffffffffu;  // layer * n_tokens + token of the cached entry
  const __half* src0 = nullptr;
  long long vid0 = -1;
};

__device__ __forceinline__ Loc locate(const EncArgs& a, uint32_t gv, TokenCache& c, int lane) {
  const uint32_t lt = fdiv(gv, a.div_h);
  const uint32_t h = gv - lt * (uint32_t)a.view.H;
  if (lt != c.lt) {
    c.lt = lt;
    const uint32_t l = fdiv(lt, a.div_t);
    const uint32_t t = lt - l * (uint32_t)a.n_tokens;
    c.src0 = a.x + (long long)l * a.layer_stride + (long long)t * a.token_stride;
    const long long slot = a.slots ? a.slots[t] : a.slot_begin + t;
    const DevView& V = a.view;
    const long long cap = V.num_pages * (long long)V.page_size;
    if (slot < 0 || slot >= cap) {
      if (lane == 0) atomicOr(a.tab.status, kFlagSlot);
      c.vid0 = -1;
    } else {
      long long page, p;
      if (a.slot32) {
        const uint32_t s32 = (uint32_t)slot, pg = fdiv(s32, a.div_p);
        page = pg;
        p = s32 - pg * (uint32_t)V.page_size;
      } else {
        page = slot / V.page_size;
        p = slot - page * V.page_size;
      }
      c.vid0 = (((long long)(a.layer_begin + (int)l) * V.num_pages + page) * V.H) * V.page_size + p;
    }
  }
  Loc r;
  r.src = c.src0 + (long long)h * a.view.d;
  r.vid = c.vid0 < 0 ? -1 : c.vid0 + (long long)h * a.view.page_size;
  return r;
}

// Raw fp16 coordinates of one lane (E = D/32 halves), loaded ahead of their use.
template <int D>
struct RawVec {
  static constexpr int E = D / 32;
  uint32_t w[E / 2];
  __device__ __forceinline__ void load(const __half* src, int lane) {
    const __half* p = src + E * lane;
    if constexpr (E == 2) {
      w[0] = *reinterpret_cast<const uint32_t*>(p);
    } else if constexpr (E == 4) {
      const uint2 u = *reinterpret_cast<const uint2*>(p);
      w[0] = u.x; w[1] = u.y;
    } else {
      const uint4 u = *reinterpret_cast<const uint4*>(p);
      w[0] = u.x; w[1] = u.y; w[2] = u.z; w[3] = u.w;
    }
  }
  __device__ __forceinline__ void zero() {
#pragma unroll
    for (int k = 0; k < E / 2; ++k) w[k] = 0u;
  }
  __device__ __forceinline__ void to_float(float (&x)[E]) const {
#pragma unroll
    for (int k = 0; k < E / 2; ++k) {
      const __half2 h = *reinterpret_cast<const __half2*>(&w[k]);
      x[2 * k] = __low2float(h);
      x[2 * k + 1] = __high2float(h);
    }
  }
};

// Spreads bits 0..3 of x to bits 0, 2, 4, 6.
__device__ __forceinline__ uint32_t spread4(uint32_t x) {
  x = (x | (x << 2)) & 0x33u;
  return (x | (x << 1)) & 0x55u;
}

// Per-lane constants of stage 1: sign flips of the lane's coordinates and the
// butterfly signs of the five shuffle stages (-1 on the upper lane of a pair).
template <int D>
struct Stage1Consts {
  float sgn[D / 32];
  float bfly[5];
  __device__ __forceinline__ void init(const int8_t* signs, int lane) {
    constexpr int E = D / 32;
#pragma unroll
    for (int e = 0; e < E; ++e) sgn[e] = (float)signs[E * lane + e];
#pragma unroll
    for (int s = 0; s < 5; ++s) bfly[s] = (lane >> s) & 1 ? -1.f : 1.f;
  }
};

// Stage 1 for one vector held by a warp: returns n and leaves y = H diag(s) x / n in x
// (orthonormal H: the butterflies run unscaled and 1/(n sqrt(d)) is applied once).
template <int D>
__device__ __forceinline__ float stage1_rotate(float (&x)[D / 32], const Stage1Consts<D>& c) {
  constexpr int E = D / 32;
  float ss = 0.f;
#pragma unroll
  for (int e = 0; e < E; ++e) {
    ss = fmaf(x[e], x[e], ss);
    x[e] *= c.sgn[e];
  }
#pragma unroll
  for (int s = 1; s < E; s <<= 1) {
#pragma unroll
    for (int i = 0; i < E; ++i) {
      if ((i & s) == 0) {
        const float u = x[i], v = x[i + s];
        x[i] = u + v;
        x[i + s] = u - v;
      }
    }
  }
  ss = warp_sum(ss);
#pragma unroll
  for (int st = 0; st < 5; ++st) {
#pragma unroll
    for (int i = 0; i < E; ++i) {
      const float o = __shfl_xor_sync(kFull, x[i], 1 << st);
      x[i] = fmaf(x[i], c.bfly[st], o);  // lower lane: x + o, upper lane: o - x
    }
  }
  const float n = sqrtf(ss);
  const float f = n > 0.f ? __fdividef(inv_sqrt_dim<D>(), n) : 0.f;  // ~2 ulp: far inside the code band
#pragma unroll
  for (int e = 0; e < E; ++e) x[e] *= f;
  return n;
}

// Lloyd-Max index of y: the number of sorted boundaries bnd[k] <= y (b bits, 2^b - 1 boundaries).
template <int B>
__device__ __forceinline__ uint32_t lloyd_index(float y, const float (&bnd)[7]) {
  if constexpr (B == 1) {
    return y >= bnd[0] ? 1u : 0u;
  } else if constexpr (B == 2) {
    const bool s1 = y >= bnd[1];
    const float t0 = s1 ? bnd[2] : bnd[0];
    return (s1 ? 2u : 0u) + (y >= t0 ? 1u : 0u);
  } else {
    const bool s2 = y >= bnd[3];
    const float t1 = s2 ? bnd[5] : bnd[1];
    const bool s1 = y >= t1;
    const float u = s2 ? bnd[4] : bnd[0], v = s2 ? bnd[6] : bnd[2];
    const float t0 = s1 ? v : u;
    return (s2 ? 4u : 0u) + (s1 ? 2u : 0u) + (y >= t0 ? 1u : 0u);
  }
}

// Stores the packed stream of one vector: lane l holds the E = D/32 codes of its
// coordinates as chunk = sum_e code_e << (W e) (bits [C l, C l + C) of the stream,
// C = E W); lane j < E W writes 32-bit word j.
template <int D, int W>
__device__ __forceinline__ void pack_store(uint32_t chunk, uint32_t* dst, int lane) {
  constexpr int E = D / 32, C = E * W, NW = E * W;
  constexpr int MAXL = (32 + C - 1) / C + 1;
  const int lfirst = (32 * lane) / C;
  uint32_t word = 0;
#pragma unroll
  for (int k = 0; k < MAXL; ++k) {
    const int src = lfirst + k;
    const uint32_t v = __shfl_sync(kFull, chunk, src & 31);
    const int sh = C * src - 32 * lane;
    if (src < 32 && sh < 32) word |= sh >= 0 ? (v << sh) : (v >> -sh);
  }
  if (lane < NW) dst[lane] = word;
}

__device__ __forceinline__ uint32_t h2u(__half2 h) { return *reinterpret_cast<uint32_t*>(&h); }

__device__ __forceinline__ void mma_16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// High and low fp16 parts of a float pair (low element in the low half).
__device__ __forceinline__ void split_pair(float2 v, uint32_t& hi, uint32_t& lo) {
  const __half2 h = __floats2half2_rn(v.x, v.y);
  const float2 hf = __half22float2(h);
  hi = h2u(h);
  lo = h2u(__floats2half2_rn(v.x - hf.x, v.y - hf.y));
}

// B = stage-1 index bits (turbo K: the stored code adds the QJL sign as bit B).
template <int D, int KIND, int B>
__global__ void __launch_bounds__(kEncThreads, KIND == kTurboK ? 3 : 4) encode_kernel(EncArgs a) {
  using Sh = EncShape<D>;
  constexpr int E = Sh::E;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;

  extern __shared__ __align__(16) unsigned char smem[];
  float* cb_s = reinterpret_cast<float*>(smem);  // centroids [8]
  unsigned char* dyn = smem + 64;

  const DevView& V = a.view;
  Stage1Consts<D> c1;
  float bnd[7];
  if (KIND == kTurboK || KIND == kTurboV) {
    c1.init(a.tab.signs, lane);
#pragma unroll
    for (int k = 0; k < 7; ++k) bnd[k] = k < (1 << B) - 1 ? a.tab.boundaries[(B - 1) * 7 + k] : 0.f;
    if (threadIdx.x < 8) cb_s[threadIdx.x] = a.tab.centroids[(B - 1) * 8 + threadIdx.x];
  }
  __syncthreads();
  TokenCache tc;

  if constexpr (KIND == kTurboK) {
    constexpr int NV = Sh::NV, RS = Sh::RS, KS = Sh::KS, W = B + 1;
    constexpr int VPW = NV / kEncWarps;                                    // vectors per warp in phases A, C
    float* r_s = reinterpret_cast<float*>(dyn);                            // [NV][RS] residual x kRScale
    uint32_t* chunk_s = reinterpret_cast<uint32_t*>(dyn + NV * RS * 4);    // [NV][32] index chunks
    uint32_t* sig_s = chunk_s + NV * 32;                                   // [NV][D/32] QJL sign bits
    long long* vid_s = reinterpret_cast<long long*>(sig_s + NV * (D / 32));  // [NV]
    const long long n_batches = (a.n_vectors + NV - 1) / NV;
    for (long long bt = blockIdx.x; bt < n_batches; bt += gridDim.x) {
      const long long base = bt * NV + warp * VPW;
      // ---- phase A: stage 1 and the residual, one warp per vector (next vector's load in flight) ----
      Loc cur{nullptr, -1};
      RawVec<D> raw;
      raw.zero();
      if (base < a.n_vectors) {
        cur = locate(a, (uint32_t)base, tc, lane);
        if (cur.vid >= 0) raw.load(cur.src, lane);
      }
#pragma unroll 1
      for (int i = 0; i < VPW; ++i) {
        const int v = warp * VPW + i;
        Loc nxt{nullptr, -1};
        RawVec<D> rawn;
        rawn.zero();
        if (i + 1 < VPW && base + i + 1 < a.n_vectors) {
          nxt = locate(a, (uint32_t)(base + i + 1), tc, lane);
          if (nxt.vid >= 0) rawn.load(nxt.src, lane);
        }
        float x[E];
        raw.to_float(x);
        const float n = stage1_rotate<D>(x, c1);
        float rr = 0.f;
        uint32_t chunk = 0;
#pragma unroll
        for (int e = 0; e < E; ++e) {
          const uint32_t idx = lloyd_index<B>(x[e], bnd);
          const float r = x[e] - cb_s[idx];
          rr = fmaf(r, r, rr);
          x[e] = r * kRScale;
          chunk |= idx << (W * e);
        }
        float* rp = r_s + v * RS + E * lane;
        if constexpr (E == 2) {
          *reinterpret_cast<float2*>(rp) = make_float2(x[0], x[1]);
        } else {
          *reinterpret_cast<float4*>(rp) = make_float4(x[0], x[1], x[2], x[3]);
          if constexpr (E == 8) *reinterpret_cast<float4*>(rp + 4) = make_float4(x[4], x[5], x[6], x[7]);
        }
        chunk_s[v * 32 + lane] = chunk;
        const float rnorm = n * sqrtf(warp_sum(rr));
        if (lane == 0) {
          vid_s[v] = cur.vid;
          if (cur.vid >= 0) {
            const __half2 hd = __halves2half2(__float2half_rn(n), __float2half_rn(rnorm));
            *reinterpret_cast<__half2*>(V.header + cur.vid * V.hdr_bytes) = hd;
          }
        }
        cur = nxt;
        raw = rawn;
      }
      __syncthreads();
      // ---- phase B: sigma_j = [(S r)_j > 0] for the batch on tensor cores ----
      // warp: vectors [16 mt, 16 mt + 16) x projections [64 pg, 64 pg + 64)
      {
        constexpr int MT = NV / 16;
        const int mt = warp % MT, pg = warp / MT;
        const int g = lane >> 2, t = lane & 3;
        float acc[8][4];
#pragma unroll
        for (int nb = 0; nb < 8; ++nb) acc[nb][0] = acc[nb][1] = acc[nb][2] = acc[nb][3] = 0.f;
        const float* ra = r_s + (16 * mt + g) * RS + 2 * t;
        const uint4* sf = a.tab.S_frag + (size_t)(8 * pg) * KS * 32 + lane;
#pragma unroll 1
        for (int ks = 0; ks < KS; ++ks) {
          uint32_t ahi[4], alo[4];
          split_pair(*reinterpret_cast<const float2*>(ra + 16 * ks), ahi[0], alo[0]);
          split_pair(*reinterpret_cast<const float2*>(ra + 8 * RS + 16 * ks), ahi[1], alo[1]);
          split_pair(*reinterpret_cast<const float2*>(ra + 16 * ks + 8), ahi[2], alo[2]);
          split_pair(*reinterpret_cast<const float2*>(ra + 8 * RS + 16 * ks + 8), ahi[3], alo[3]);
#pragma unroll
          for (int nb = 0; nb < 8; ++nb) {
            const uint4 b = __ldg(sf + ((size_t)nb * KS + ks) * 32);
            mma_16816(acc[nb], alo, b.x, b.y);
            mma_16816(acc[nb], ahi, b.z, b.w);
            mma_16816(acc[nb], ahi, b.x, b.y);
          }
        }
        // sign bits by ballot: bit (4g + t) of ballot c of block nb is the sign of
        // c0: (vector g, projection 8nb + 2t), c1: (g, 2t + 1), c2: (g + 8, 2t), c3: (g + 8, 2t + 1)
        // lane: vector vv of the tile, projections 32 half + [0, 32) of the warp's 64
        const int vv = lane & 15, half = lane >> 4, gg = vv & 7;
        const bool upper = vv >= 8;
        uint32_t word = 0;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          uint32_t b0[4], b1[4];  // ballots of blocks q and 4 + q
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            b0[c] = __ballot_sync(kFull, acc[q][c] > 0.f);
            b1[c] = __ballot_sync(kFull, acc[4 + q][c] > 0.f);
          }
          const uint32_t be = half ? (upper ? b1[2] : b1[0]) : (upper ? b0[2] : b0[0]);
          const uint32_t bo = half ? (upper ? b1[3] : b1[1]) : (upper ? b0[3] : b0[1]);
          const uint32_t byte = spread4((be >> (4 * gg)) & 15u) | (spread4((bo >> (4 * gg)) & 15u) << 1);
          word |= byte << (8 * q);
        }
        sig_s[(16 * mt + vv) * (D / 32) + 2 * pg + half] = word;
      }
      __syncthreads();
      // ---- phase C: codes = index | sign << B, pack and store ----
#pragma unroll 1
      for (int i = 0; i < VPW; ++i) {
        const int v = warp * VPW + i;
        const long long vid = vid_s[v];
        if (vid < 0) continue;  // warp-uniform
        const uint32_t sbits = (sig_s[v * (D / 32) + (E * lane) / 32] >> ((E * lane) % 32)) & ((1u << E) - 1u);
        uint32_t chunk = chunk_s[v * 32 + lane];
#pragma unroll
        for (int e = 0; e < E; ++e) chunk |= ((sbits >> e) & 1u) << (W * e + B);
        pack_store<D, W>(chunk, reinterpret_cast<uint32_t*>(V.payload + vid * V.pay_bytes), lane);
      }
      __syncthreads();
    }
  } else {
    // warps take runs of 8 consecutive vectors (whole tokens when H divides 8), the next
    // vector's load in flight while the current one is encoded
    uint8_t* codes_s = dyn + warp * D;  // [warps][D] (min-max packing)
    constexpr int RUN = 8;
    const long long nw = (long long)gridDim.x * kEncWarps;
    long long run = (long long)blockIdx.x * kEncWarps + warp;
    int i = 0;
    long long gv = run * RUN;
    Loc cur{nullptr, -1};
    RawVec<D> raw;
    raw.zero();
    if (gv < a.n_vectors) {
      cur = locate(a, (uint32_t)gv, tc, lane);
      if (cur.vid >= 0) raw.load(cur.src, lane);
    }
    while (gv < a.n_vectors) {
      // next vector of this warp
      long long gn;
      if (i + 1 < RUN) {
        gn = gv + 1;
        ++i;
      } else {
        run += nw;
        gn = run * RUN;
        i = 0;
      }
      Loc nxt{nullptr, -1};
      RawVec<D> rawn;
      rawn.zero();
      if (gn < a.n_vectors) {
        nxt = locate(a, (uint32_t)gn, tc, lane);
        if (nxt.vid >= 0) rawn.load(nxt.src, lane);
      }
      if (cur.vid >= 0) {  // warp-uniform
        float x[E];
        raw.to_float(x);
        unsigned char* pay = V.payload + cur.vid * V.pay_bytes;
        unsigned char* hdr = V.header + cur.vid * V.hdr_bytes;
        if constexpr (KIND == kTurboV) {
          const float n = stage1_rotate<D>(x, c1);
          uint32_t chunk = 0;
#pragma unroll
          for (int e = 0; e < E; ++e) chunk |= lloyd_index<B>(x[e], bnd) << (B * e);
          if (lane == 0) *reinterpret_cast<__half*>(hdr) = __float2half_rn(n);
          pack_store<D, B>(chunk, reinterpret_cast<uint32_t*>(pay), lane);
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
          const int b = V.idx_bits;
          const int qmax = (1 << b) - 1;
          const float scale = __fdiv_rn(__fsub_rn(mx, mn), (float)qmax);
#pragma unroll
          for (int e = 0; e < E; ++e) {
            int q = 0;
            if (scale > 0.f) {
              const float tq = __fadd_rn(__fdiv_rn(__fsub_rn(x[e], mn), scale), 0.5f);
              q = (int)floorf(tq);
              q = q < 0 ? 0 : (q > qmax ? qmax : q);
            }
            codes_s[E * lane + e] = (uint8_t)q;
          }
          if ((lane % (64 / E)) == 0)
            reinterpret_cast<__half2*>(hdr)[lane / (64 / E)] =
                __halves2half2(__float2half_rn(scale), __float2half_rn(mn));
          __syncwarp();
          warp_pack_store<D>(codes_s, V.code_bits, reinterpret_cast<uint32_t*>(pay), lane);
          __syncwarp();
        }
      }
      cur = nxt;
      raw = rawn;
      gv = gn;
    }
  }
}

template <int D, int KIND, int B>
cudaError_t launch_kind(const EncArgs& a, int sm_count, cudaStream_t s) {
  size_t smem = 64;
  long long work;
  if (KIND == kTurboK) {
    using Sh = EncShape<D>;
    smem += (size_t)Sh::NV * Sh::RS * 4 + (size_t)Sh::NV * 32 * 4 + (size_t)Sh::NV * (D / 32) * 4 + Sh::NV * 8;
    work = (a.n_vectors + Sh::NV - 1) / Sh::NV;
  } else {
    smem += (size_t)kEncWarps * D;
    work = (a.n_vectors + 8 * kEncWarps - 1) / (8 * kEncWarps);  // runs of 8 vectors per warp
  }
  auto kern = encode_kernel<D, KIND, B>;
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

template <int D, int KIND>
cudaError_t launch_bits(const EncArgs& a, int sm_count, cudaStream_t s) {
  switch (a.view.idx_bits) {
    case 1: return launch_kind<D, KIND, 1>(a, sm_count, s);
    case 2: return launch_kind<D, KIND, 2>(a, sm_count, s);
    case 3: return launch_kind<D, KIND, 3>(a, sm_count, s);
  }
  return cudaErrorInvalidValue;
}

template <int D>
cudaError_t launch_dim(const EncArgs& a, int sm_count, cudaStream_t s) {
  const int f = a.view.format;
  if (f == TQ_FMT_Q8_0) return launch_kind<D, kQ8, 1>(a, sm_count, s);
  if (f == TQ_FMT_MINMAX) return launch_kind<D, kMinMax, 1>(a, sm_count, s);
  if (a.view.has_qjl) return launch_bits<D, kTurboK>(a, sm_count, s);
  return launch_bits<D, kTurboV>(a, sm_count, s);
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
  a.div_h = make_fastdiv((uint32_t)view.H);
  a.div_t = make_fastdiv((uint32_t)n_tokens);
  const long long cap = view.num_pages * (long long)view.page_size;
  a.slot32 = cap <= 0xffffffffLL ? 1 : 0;
  a.div_p = make_fastdiv((uint32_t)view.page_size);
  switch (view.d) {
    case 64: return launch_dim<64>(a, sm_count, s);
    case 128: return launch_dim<128>(a, sm_count, s);
    case 256: return launch_dim<256>(a, sm_count, s);
  }
  return cudaErrorInvalidValue;
}

}  // namespace tq
