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
//   - turbo formats at d = 128: encode_tc_kernel (tensor cores; described at the kernel).
//     The Lloyd-Max index there is step_count_signed, a sum of saturated FMA steps on |y|
//     that equals the count of boundaries <= y (an exact tie at a negative boundary,
//     measure zero, takes the lower index);
//   - turbo formats at d = 64 and 256: a vector is held by a group of L = d/32 lanes,
//     each lane owning 32 consecutive coordinates, so a warp encodes 32/L vectors at
//     once.  The sign flips are applied on the fp16 words, five of the WHT stages run
//     inside a lane and log2(L) across the group (shuffles), 1/(n sqrt(d)) is applied
//     once; the Lloyd-Max index is a binary search over the sorted boundaries (the
//     count of boundaries <= y, ties included as the definition has it), and each lane
//     packs its 32 codes into its own w words of the stream and stores them;
//   - turbo K at d = 64 / 256: a CTA encodes a batch of NV = 8192/d vectors: phase A (stage 1, the
//     residual r into shared memory), phase B (the whole CTA: the d x d projection
//     S r on mma.sync m16n8k16, f16 inputs split into high and low parts,
//     r_hi s_hi + r_lo s_hi + r_hi s_lo accumulated in fp32, which leaves an error
//     near 1e-7 of |r|, far inside the 1e-6 sign band; signs gathered by warp
//     ballots), phase C (codes = index | sign << b, stored);
//   - q8_0 and min-max: one warp per vector, lane l holds E = d/32 coordinates;
//   - vector ids -> (layer, token, head) and slots -> (page, offset) use
//     multiply-shift division by invariant divisors;
//   - grids are persistent: min(work, resident CTAs) CTAs loop over the work.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_fp16.h>

#include "tq_device.cuh"
#include "tq_tc.cuh"

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

// The same split with the subtraction in packed fp32.
__device__ __forceinline__ void split_pair2(float2 v, uint32_t& hi, uint32_t& lo) {
  const __half2 h = __floats2half2_rn(v.x, v.y);
  const float2 hf = __half22float2(h);
  hi = h2u(h);
  const float2 d = __ffma2_rn(hf, make_float2(-1.f, -1.f), v);
  lo = h2u(__floats2half2_rn(d.x, d.y));
}

// q8_0 and per-group min-max: one warp per vector (lane l holds E = d/32 coordinates).
template <int D, int KIND>
__global__ void __launch_bounds__(kEncThreads, 4) encode_kernel(EncArgs a) {
  constexpr int E = D / 32;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  extern __shared__ __align__(16) unsigned char smem[];
  uint8_t* codes_s = smem + warp * D;  // [warps][D] (min-max packing)
  const DevView& V = a.view;
  TokenCache tc;
  // warps take runs of 8 consecutive vectors (whole tokens when H divides 8), the next
  // vector's load in flight while the current one is encoded
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
      if constexpr (KIND == kQ8) {
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

// ---------------------------------------------------------------------------
// Turbo formats: a vector is held by a group of L = d/32 lanes, each lane owning 32
// consecutive coordinates, so a warp encodes 32/L vectors at once.  Five of the WHT
// stages, the Lloyd-Max indices and the packing of the lane's own code words stay in
// registers; only log2(L) butterfly stages and the norm need shuffles within the group.
// ---------------------------------------------------------------------------
template <int D>
struct GroupShape {
  static constexpr int L = D / 32;       // lanes per vector
  static constexpr int VPW = 32 / L;     // vectors per warp
  static constexpr int NV = 8192 / D;    // vectors per CTA batch (turbo K) = warps x VPW
  static constexpr int RS = D + 8;       // row stride of the residual tile (floats)
  static constexpr int KS = D / 16;      // k steps of the projection
  static_assert(NV == kEncWarps * VPW, "one group pass per warp and batch");
};

// Residual tile swizzle: the 16-byte chunk k (coordinates 32 sub + 4k .. + 3) of a row is
// stored at chunk k ^ f(sub), so that the 8 lanes of a 128-bit store (consecutive lanes
// covering 2 rows of 4 groups at d = 128) fall on 8 distinct 4-bank groups; the projection's
// 64-bit loads use the same map and stay conflict-free.
template <int L>
__device__ __forceinline__ int chunk_swz(int sub) {
  return L == 4 ? ((sub & 1) | ((sub & 2) << 1)) : sub;
}
// Swizzled position (in floats) of coordinate c in a residual row.
template <int L>
__device__ __forceinline__ int r_pos(int c) {
  const int sub = c >> 5;
  return (c & ~31) | ((((c >> 2) & 7) ^ chunk_swz<L>(sub)) << 2) | (c & 3);
}

// fp16 sign masks of the lane's 32 coordinates: word j flips coordinates 2j, 2j+1.
__device__ __forceinline__ void lane_sign_masks(const int8_t* signs, int sub, uint32_t (&sg)[16]) {
#pragma unroll
  for (int j = 0; j < 16; ++j)
    sg[j] = (signs[32 * sub + 2 * j] < 0 ? 0x8000u : 0u) | (signs[32 * sub + 2 * j + 1] < 0 ? 0x80000000u : 0u);
}

// The lane's 32 fp16 coordinates (64 contiguous bytes), loaded ahead of their use.
struct Raw32 {
  uint4 q[4];
  __device__ __forceinline__ void load(const __half* src) {
    const uint4* p = reinterpret_cast<const uint4*>(src);
#pragma unroll
    for (int k = 0; k < 4; ++k) q[k] = p[k];
  }
  __device__ __forceinline__ void zero() {
#pragma unroll
    for (int k = 0; k < 4; ++k) q[k] = make_uint4(0u, 0u, 0u, 0u);
  }
  // signs applied on the fp16 words (exact), then widened to fp32
  __device__ __forceinline__ void to_float(float (&x)[32], const uint32_t (&sg)[16]) const {
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const uint32_t w[4] = {q[k].x, q[k].y, q[k].z, q[k].w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint32_t u = w[i] ^ sg[4 * k + i];
        const __half2 h = *reinterpret_cast<const __half2*>(&u);
        x[8 * k + 2 * i] = __low2float(h);
        x[8 * k + 2 * i + 1] = __high2float(h);
      }
    }
  }
};

// Stage 1 of one vector held by a group: x holds diag(s) x on entry (coordinates 32 sub + e);
// returns n and leaves y = H diag(s) x / n.  The butterflies run unscaled and 1/(n sqrt(d)) is
// applied once; bfly[s] = -1 on the upper lane of each pair of the cross-lane stage s.
template <int D>
__device__ __forceinline__ float group_stage1(float (&x)[32], const float (&bfly)[3]) {
  constexpr int L = D / 32;
  float ss = 0.f;
#pragma unroll
  for (int e = 0; e < 32; ++e) ss = fmaf(x[e], x[e], ss);  // |s_i x_i| = |x_i|
#pragma unroll
  for (int s = 1; s < 32; s <<= 1) {
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      if ((i & s) == 0) {
        const float u = x[i], v = x[i + s];
        x[i] = u + v;
        x[i + s] = u - v;
      }
    }
  }
#pragma unroll
  for (int m = 1; m < L; m <<= 1) ss += __shfl_xor_sync(kFull, ss, m);
#pragma unroll
  for (int st = 0; (1 << st) < L; ++st) {
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      const float o = __shfl_xor_sync(kFull, x[i], 1 << st);
      x[i] = fmaf(x[i], bfly[st], o);  // lower lane: x + o, upper lane: o - x
    }
  }
  const float n = sqrtf(ss);
  const float f = n > 0.f ? __fdividef(inv_sqrt_dim<D>(), n) : 0.f;  // ~2 ulp: far inside the code band
#pragma unroll
  for (int e = 0; e < 32; ++e) x[e] *= f;
  return n;
}

// ORs the W-bit code c of the lane's coordinate e into its W words (bit W e of the lane's stream).
template <int W>
__device__ __forceinline__ void put_code(uint32_t (&w)[W], int e, uint32_t c) {
  const int bit = W * e, k = bit >> 5, sh = bit & 31;
  w[k] |= c << sh;
  if (sh + W > 32) w[k + 1] |= c >> (32 - sh);
}

// Stores the lane's W words at word W sub of the vector's payload.
template <int W>
__device__ __forceinline__ void store_words(uint32_t* dst, const uint32_t (&w)[W]) {
  if constexpr (W == 4) {
    *reinterpret_cast<uint4*>(dst) = make_uint4(w[0], w[1], w[2], w[3]);
  } else if constexpr (W == 2) {
    *reinterpret_cast<uint2*>(dst) = make_uint2(w[0], w[1]);
  } else {
#pragma unroll
    for (int k = 0; k < W; ++k) dst[k] = w[k];
  }
}

// Location of the vector of global id gv (no caching: the lanes of a warp serve different vectors).
__device__ __forceinline__ Loc locate_one(const EncArgs& a, uint32_t gv, int report) {
  const uint32_t lt = fdiv(gv, a.div_h);
  const uint32_t h = gv - lt * (uint32_t)a.view.H;
  const uint32_t l = fdiv(lt, a.div_t);
  const uint32_t t = lt - l * (uint32_t)a.n_tokens;
  Loc r;
  r.src = a.x + (long long)l * a.layer_stride + (long long)t * a.token_stride + (long long)h * a.view.d;
  const long long slot = a.slots ? a.slots[t] : a.slot_begin + t;
  const DevView& V = a.view;
  const long long cap = V.num_pages * (long long)V.page_size;
  if (slot < 0 || slot >= cap) {
    if (report && h == 0) atomicOr(a.tab.status, kFlagSlot);
    r.vid = -1;
    return r;
  }
  long long page, p;
  if (a.slot32) {
    const uint32_t s32 = (uint32_t)slot, pg = fdiv(s32, a.div_p);
    page = pg;
    p = s32 - pg * (uint32_t)V.page_size;
  } else {
    page = slot / V.page_size;
    p = slot - page * V.page_size;
  }
  r.vid = (((long long)(a.layer_begin + (int)l) * V.num_pages + page) * V.H + h) * V.page_size + p;
  return r;
}

// B = stage-1 index bits; QJL: turbo K (code = index | sign << B, plus residual norm).
template <int D, bool QJL, int B>
__global__ void __launch_bounds__(kEncThreads, 2) encode_turbo_kernel(EncArgs a) {
  using Sh = GroupShape<D>;
  constexpr int L = Sh::L, VPW = Sh::VPW;
  constexpr int W = QJL ? B + 1 : B;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int sub = lane % L, vl = lane / L;

  extern __shared__ __align__(16) unsigned char smem[];
  float* cb_s = reinterpret_cast<float*>(smem);  // centroids [8]
  unsigned char* dyn = smem + 64;
  if (threadIdx.x < 8) cb_s[threadIdx.x] = a.tab.centroids[(B - 1) * 8 + threadIdx.x];

  uint32_t sg[16];
  lane_sign_masks(a.tab.signs, sub, sg);
  float bfly[3];
#pragma unroll
  for (int s = 0; s < 3; ++s) bfly[s] = (sub >> s) & 1 ? -1.f : 1.f;
  float bnd[7];
#pragma unroll
  for (int k = 0; k < 7; ++k) bnd[k] = k < (1 << B) - 1 ? a.tab.boundaries[(B - 1) * 7 + k] : 0.f;
  __syncthreads();
  const DevView& V = a.view;

  if constexpr (QJL) {
    constexpr int NV = Sh::NV, RS = Sh::RS, KS = Sh::KS;
    float* r_s = reinterpret_cast<float*>(dyn);                              // [NV][RS] residual x kRScale
    uint32_t* code_s = reinterpret_cast<uint32_t*>(dyn + NV * RS * 4);      // [NV][L][W] index words
    uint32_t* sig_s = code_s + NV * L * W;                                  // [NV][D/32] QJL sign bits
    long long* vid_s = reinterpret_cast<long long*>(sig_s + NV * (D / 32));  // [NV]
    const long long n_batches = (a.n_vectors + NV - 1) / NV;
    for (long long bt = blockIdx.x; bt < n_batches; bt += gridDim.x) {
      const int v = warp * VPW + vl;  // this lane's vector in the batch
      const long long gv = bt * NV + v;
      // ---- phase A: stage 1 and the residual ----
      {
        Loc loc{nullptr, -1};
        Raw32 raw;
        raw.zero();
        if (gv < a.n_vectors) {
          loc = locate_one(a, (uint32_t)gv, sub == 0);
          if (loc.vid >= 0) raw.load(loc.src + 32 * sub);
        }
        float x[32];
        raw.to_float(x, sg);
        const float n = group_stage1<D>(x, bfly);
        float rr = 0.f;
        uint32_t w[W] = {};
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          const uint32_t idx = lloyd_index<B>(x[e], bnd);
          const float r = x[e] - cb_s[idx];
          rr = fmaf(r, r, rr);
          x[e] = r * kRScale;
          put_code<W>(w, e, idx);
        }
        float4* rp = reinterpret_cast<float4*>(r_s + v * RS + 32 * sub);
        const int swz = chunk_swz<L>(sub);
#pragma unroll
        for (int k = 0; k < 8; ++k) rp[k ^ swz] = make_float4(x[4 * k], x[4 * k + 1], x[4 * k + 2], x[4 * k + 3]);
        uint32_t* cw = code_s + (v * L + sub) * W;
#pragma unroll
        for (int k = 0; k < W; ++k) cw[k] = w[k];
#pragma unroll
        for (int m = 1; m < L; m <<= 1) rr += __shfl_xor_sync(kFull, rr, m);
        const float rnorm = n * sqrtf(rr);
        if (sub == 0) {
          vid_s[v] = loc.vid;
          if (loc.vid >= 0)
            *reinterpret_cast<__half2*>(V.header + loc.vid * V.hdr_bytes) =
                __halves2half2(__float2half_rn(n), __float2half_rn(rnorm));
        }
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
        const float* ra = r_s + (16 * mt + g) * RS;
        const uint4* sf = a.tab.S_frag + (size_t)(8 * pg) * KS * 32 + lane;
#pragma unroll 1
        for (int ks = 0; ks < KS; ++ks) {
          uint32_t ahi[4], alo[4];
          const int c0 = r_pos<L>(16 * ks + 2 * t), c1 = r_pos<L>(16 * ks + 2 * t + 8);
          split_pair(*reinterpret_cast<const float2*>(ra + c0), ahi[0], alo[0]);
          split_pair(*reinterpret_cast<const float2*>(ra + 8 * RS + c0), ahi[1], alo[1]);
          split_pair(*reinterpret_cast<const float2*>(ra + c1), ahi[2], alo[2]);
          split_pair(*reinterpret_cast<const float2*>(ra + 8 * RS + c1), ahi[3], alo[3]);
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
      // ---- phase C: codes = index | sign << B, store ----
      {
        const long long vid = vid_s[v];
        if (vid >= 0) {
          uint32_t w[W];
          const uint32_t* cw = code_s + (v * L + sub) * W;
#pragma unroll
          for (int k = 0; k < W; ++k) w[k] = cw[k];
          const uint32_t sbits = sig_s[v * (D / 32) + sub];
          if constexpr (W == 4) {
            // bits 8k..8k+7 of sbits -> bit 3 of each nibble of word k
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              uint32_t b = (sbits >> (8 * k)) & 0xFFu;
              b = (b | (b << 12)) & 0x000F000Fu;
              b = (b | (b << 6)) & 0x03030303u;
              b = (b | (b << 3)) & 0x11111111u;
              w[k] |= b << 3;
            }
          } else {
#pragma unroll
            for (int e = 0; e < 32; ++e) {
              const int bit = W * e + B;
              w[bit >> 5] |= ((sbits >> e) & 1u) << (bit & 31);
            }
          }
          store_words<W>(reinterpret_cast<uint32_t*>(V.payload + vid * V.pay_bytes) + W * sub, w);
        }
      }
      __syncthreads();
    }
  } else {
    // V: warps take groups of VPW consecutive vectors; the next group's loads are in flight
    // while the current one is encoded
    const long long nw = (long long)gridDim.x * kEncWarps;
    long long grp = (long long)blockIdx.x * kEncWarps + warp;
    long long gv = grp * VPW + vl;
    Loc cur{nullptr, -1};
    Raw32 raw;
    raw.zero();
    if (gv < a.n_vectors) {
      cur = locate_one(a, (uint32_t)gv, sub == 0);
      if (cur.vid >= 0) raw.load(cur.src + 32 * sub);
    }
    while (grp * VPW < a.n_vectors) {  // warp-uniform
      const long long gn = gv + nw * VPW;
      Loc nxt{nullptr, -1};
      Raw32 rawn;
      rawn.zero();
      if (gn < a.n_vectors) {
        nxt = locate_one(a, (uint32_t)gn, sub == 0);
        if (nxt.vid >= 0) rawn.load(nxt.src + 32 * sub);
      }
      float x[32];
      raw.to_float(x, sg);
      const float n = group_stage1<D>(x, bfly);
      if (cur.vid >= 0) {
        uint32_t w[W] = {};
#pragma unroll
        for (int e = 0; e < 32; ++e) put_code<W>(w, e, lloyd_index<B>(x[e], bnd));
        store_words<W>(reinterpret_cast<uint32_t*>(V.payload + cur.vid * V.pay_bytes) + W * sub, w);
        if (sub == 0) *reinterpret_cast<__half*>(V.header + cur.vid * V.hdr_bytes) = __float2half_rn(n);
      }
      cur = nxt;
      raw = rawn;
      gv = gn;
      grp += nw;
    }
  }
}


// ---------------------------------------------------------------------------
// Turbo K and V at d = 128 on the fifth-generation tensor cores.  One CTA per SM: 16 SIMT warps
// and issuer warps (A: tensor copies and rotations; B, turbo K only: projections).  A batch is
// the H TB vectors (TB = floor(128 / H)) of TB consecutive tokens of one layer, all heads; row r
// of a batch is token r / H, head r % H.
//   - issuer A loads batches ahead by TMA (a 4-D tensor map over (d, head, token, layer); one
//     box per 64-coordinate half, written with the 128-byte swizzle, which is the K-major
//     operand layout the tensor core reads); tokens past the end read as zero;
//   - the rotation Y = X (H D)^T runs as tcgen05.mma (M 128) into tensor memory.  H D has
//     entries +-1 (exact in fp16) and x is fp16, so only the fp32 accumulation rounds.  V keeps
//     H D whole (8 MMAs of N 128); turbo K, short of shared memory, uses the Sylvester split of
//     H_128 into H_64 blocks: y_top = H64 D_a a + H64 D_b b, y_bot = H64 D_a a - H64 D_b b, with
//     a, b the halves of x (16 MMAs of N 64);
//   - turbo K: the QJL projection P = R S^T of R = 2^14 r split into fp16 high and low parts
//     (R_lo S_hi + R_hi S_lo + R_hi S_hi); R_hi is written over the consumed input tile;
//   - the issuers run ahead of the SIMT warps: the rotation of batch j + 1 and the projection of
//     batch j overlap the SIMT work of batch j, and the sign bits of batch j are merged into its
//     words during batch j + 1.  SIMT warps report per warp on mbarriers (Y read, R stored,
//     P read) and meet each other on a named barrier, so the issuers never stop them;
//   - SIMT warp w reads tensor-memory lanes 32 (w % 4) .. + 31 (one row per thread) and
//     columns 32 (w / 4) .. + 31, so a thread finishes 32 coordinates of one vector: norm
//     (partial sums exchanged in shared memory), Lloyd-Max index, residual, sign bits, words.
// Every wait is bounded; a wait that runs out stops the CTA and sets the timeout status bit.
// ---------------------------------------------------------------------------
namespace etc {
constexpr int D = 128, NV = 128, SIMT_WARPS = 16;
// issuer warps: A (tensor copies, rotation), and for turbo K B (projection) on another SM
// sub-partition: an MMA or copy instruction waits long for an issue slot next to warps that keep
// the FMA pipe saturated, so the projection's 24 MMAs get a scheduler of their own
template <bool QJL>
constexpr int kThreads = 32 * (SIMT_WARPS + (QJL ? 2 : 1));
constexpr int kOp = D * NV * 2;  // one 128 x 128 f16 operand
constexpr int kG = 64 * 64 * 2;  // one 64 x 64 f16 block of the rotation
// Every operand tile is K-major with the 128-byte swizzle, one 64-column half after the other:
// half k/64 at 128 R (R rows), row r at 128 r, 16-byte chunk (k % 64) / 8 at chunk position
// ((k % 64) / 8) ^ (r % 8).  The tensor copy writes the input tiles in this layout.
template <int R>
__host__ __device__ constexpr int swz(int row, int k) {
  return (k >> 6) * (128 * R) + row * 128 + ((((k >> 3) & 7) ^ (row & 7)) << 4) + (k & 7) * 2;
}
// K step ks (16 columns) of a tile with R rows: start of its descriptor
template <int R>
__host__ __device__ constexpr uint32_t kstep(int ks) {
  return (uint32_t)((ks >> 2) * (128 * R) + (ks & 3) * 32);
}

template <bool QJL>
struct Smem {  // byte offsets in dynamic shared memory
  static constexpr int NX = QJL ? 3 : 4;            // input tiles in flight
  static constexpr int g = 0;                        // K: H64 D_a, H64 D_b, -H64 D_b; V: H D (128 x 128)
  static constexpr int s_hi = QJL ? 3 * kG : kOp;    // S high part (QJL)
  static constexpr int s_lo = s_hi + (QJL ? kOp : 0);
  static constexpr int x0 = s_lo + (QJL ? kOp : 0);  // NX input tiles (batch j in tile j % NX)
  static constexpr int r_lo = x0 + NX * kOp;          // R low part (QJL)
  static constexpr int NY = QJL ? 2 : 4;             // Y buffers in tensor memory
  static constexpr int ss = r_lo + (QJL ? kOp : 0);   // float [NY][4][NV]: partial sums of y^2
  static constexpr int rr = ss + NY * 4 * NV * 4;     // float [2][4][NV]: partial sums of (2^14 r)^2
  static constexpr int cb = rr + (QJL ? 2 * 4 * NV * 4 : 0);  // float [8]: centroids x -2^14 (32-byte aligned)
  static constexpr int bar = cb + 8 * 4;  // mbarriers: full[NX], y[NY], p[2], yfree[NY], rready, pfree[2]
  static constexpr int n_bar = NX + 2 * NY + 5;
  static constexpr int slot = bar + n_bar * 8;  // tensor-memory address, abort flag
  static constexpr int total = slot + 16;
};

struct TcShape {
  int H, TB, rows;      // heads, tokens per batch, rows = H TB
  uint32_t n_tb;        // token blocks per layer
  FastDiv div_tb;
  long long n_batches;  // n_layers n_tb
  uint32_t tx_bytes;    // bytes one batch's copies deliver
};

// Destination id of vector (layer l of the input, token t, head h), or -1 for a slot out of range.
__device__ __forceinline__ long long vid_at(const EncArgs& a, int l, int t, int h, bool report) {
  const long long slot = a.slots ? a.slots[t] : a.slot_begin + t;
  const DevView& V = a.view;
  const long long cap = V.num_pages * (long long)V.page_size;
  if (slot < 0 || slot >= cap) {
    if (report && h == 0) atomicOr(a.tab.status, kFlagSlot);
    return -1;
  }
  long long page, p;
  if (a.slot32) {
    const uint32_t s32 = (uint32_t)slot, pg = fdiv(s32, a.div_p);
    page = pg;
    p = s32 - pg * (uint32_t)V.page_size;
  } else {
    page = slot / V.page_size;
    p = slot - page * V.page_size;
  }
  return (((long long)(a.layer_begin + l) * V.num_pages + page) * V.H + h) * V.page_size + p;
}

// Merges the QJL sign bits (bit e of sbits: projection 32 c + e, c = the thread's column group)
// into the thread's W words: the code of coordinate e is index | sign << B at bit W e.
template <int W, int B>
__device__ __forceinline__ void merge_signs(uint32_t (&w)[W], uint32_t sbits) {
  if constexpr (W == 4) {
#pragma unroll
    for (int k = 0; k < 4; ++k) {  // bits 8k .. 8k + 7 -> bit 3 of each nibble of word k
      uint32_t b = (sbits >> (8 * k)) & 0xFFu;
      b = (b | (b << 12)) & 0x000F000Fu;
      b = (b | (b << 6)) & 0x03030303u;
      b = (b | (b << 3)) & 0x11111111u;
      w[k] |= b << 3;
    }
  } else {
#pragma unroll
    for (int e = 0; e < 32; ++e) {
      const int bit = W * e + B;
      w[bit >> 5] |= ((sbits >> e) & 1u) << (bit & 31);
    }
  }
}

// Lloyd-Max index on the FMA pipe.  With C_k = -prev(b_k) 2^100 (prev: the next float below;
// C_k = 1 for b_k = 0), sat(u 2^100 + C_k) is 1 for u >= b_k and 0 below, exactly, whenever
// u - prev(b_k) is 0 or at least 2^-100 in magnitude.  Nonzero rotated coordinates are sums of
// fp16 values scaled by 1 / (n sqrt(d)), at least 2^-24 / (65504 sqrt(d)) in magnitude, so
// this holds for every boundary that is 0 or at least 2^-60 in magnitude (checked per call, with
// the odd symmetry of the boundaries that step_count_signed relies on; the binary search runs
// where either fails).
template <int B>
__device__ __forceinline__ bool step_constants(const float (&bnd)[7], float (&cst)[7]) {
  bool ok = true;
#pragma unroll
  for (int k = 0; k < (1 << B) - 1; ++k) ok = ok && bnd[k] == -bnd[(1 << B) - 2 - k];
#pragma unroll
  for (int k = 0; k < 7; ++k) {
    const float b = bnd[k];
    if (k >= (1 << B) - 1) {
      cst[k] = 0.f;
    } else if (b == 0.f) {
      cst[k] = 1.f;
    } else {
      ok = ok && fabsf(b) >= 0x1p-60f;
      cst[k] = -nextafterf(b, -INFINITY) * 0x1p100f;
    }
  }
  return ok;
}
// The index of y (a rotated coordinate before the 1 / (n sqrt(d)) scale; F = 2^100 / (n sqrt(d))),
// for two coordinates at once, by the codebook's odd symmetry (the boundaries are b_k = -b_(2H-2-k),
// H = 2^(B-1), the middle one exactly 0): with a = |y| and cnt = #{positive boundaries <= a} (exact
// FMA steps), the index is H + cnt for y >= 0 and H - 1 - cnt below, H - 1 steps instead of 2H - 1.
// It equals the count of boundaries <= u except at an exact tie u = -b_k (measure zero), which takes
// the lower index: such a coordinate sits on a decision boundary, inside the comparison band.
// Returned as the signed count cs = +-(1/2 + cnt), the index being H - 1/2 + cs: the steps are
// scalar (saturated FMAs), their sums packed fp32 pairs (add.rn.f32x2).  The sign is that of y + 0,
// so that y = -0 takes the upper index, as y >= 0 does.
template <int B>
__device__ __forceinline__ float2 step_count_signed(float ya, float yb, float F, const float (&cst)[7]) {
  constexpr int H = 1 << (B - 1);
  float2 c = make_float2(0.5f, 0.5f);
#pragma unroll
  for (int k = 0; k < H - 1; ++k)
    c = __fadd2_rn(c, make_float2(__saturatef(fmaf(fabsf(ya), F, cst[H + k])), __saturatef(fmaf(fabsf(yb), F, cst[H + k]))));
  const float2 yz = __fadd2_rn(make_float2(ya, yb), make_float2(0.f, 0.f));
  c.x = __uint_as_float(__float_as_uint(c.x) | (__float_as_uint(yz.x) & 0x80000000u));
  c.y = __uint_as_float(__float_as_uint(c.y) | (__float_as_uint(yz.y) & 0x80000000u));
  return c;
}
// Starting value of a packed code accumulator over a chunk of CPC W-bit codes: the (H - 1/2) part
// of each index times its place 2^(W e), even e in .x and odd e in .y (exact: all below 2^24).
template <int B, int W, int CPC>
__device__ __forceinline__ float2 code_base() {
  constexpr float h = (float)(1 << (B - 1)) - 0.5f;
  float ev = 0.f, od = 0.f;
#pragma unroll
  for (int e = 0; e < CPC; ++e) {
    if (e & 1) od += h * (float)(1u << (W * e));
    else ev += h * (float)(1u << (W * e));
  }
  return make_float2(ev, od);
}
// A read of the centroid table (written once before the CTA's first barrier, constant after it).
__device__ __forceinline__ float lds_f32(uint32_t addr) {
  float v;
  asm("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(addr));
  return v;
}
// ORs an nb-bit chunk into the thread's W words at bit offset off (compile-time after unrolling).
template <int W>
__device__ __forceinline__ void or_bits(uint32_t (&w)[W], int off, int nb, uint32_t v) {
  const int k = off >> 5, sh = off & 31;
  w[k] |= v << sh;
  if (sh + nb > 32) w[k + 1] |= v >> (32 - sh);
}
}  // namespace etc

template <bool QJL, int B>
__global__ void __launch_bounds__(etc::kThreads<QJL>, 1)
    encode_tc_kernel(const __grid_constant__ EncArgs a, const __grid_constant__ CUtensorMap tmap,
                     const etc::TcShape sh) {
  using namespace etc;
  using L = Smem<QJL>;
  constexpr int NX = L::NX;
  constexpr int W = QJL ? B + 1 : B;
  constexpr int kSimt = 32 * SIMT_WARPS;
  constexpr int NY = L::NY;
  constexpr uint32_t kCols = 512;  // K: Y[2] at columns [0, 256), P[2] at [256, 512); V: Y[4]
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  constexpr int THREADS = kThreads<QJL>;
  const bool issuer = warp >= SIMT_WARPS;  // warp SIMT_WARPS: issuer A; SIMT_WARPS + 1: issuer B
  const int q = warp & 3, cg = (warp >> 2) & 3;  // tensor-memory lane quarter, column group
  const int v = 32 * q + lane;                   // this thread's row of the batch
  const int tt = v / sh.H, h = v - tt * sh.H;

  extern __shared__ __align__(16) unsigned char smem_raw[];
  // operand tiles and tensor-copy destinations on a 1024-byte boundary (1 KB extra is allocated)
  unsigned char* smem = smem_raw + ((1024u - (tc::smem_addr(smem_raw) & 1023u)) & 1023u);
  float* ss_s = reinterpret_cast<float*>(smem + L::ss);
  float* rr_s = reinterpret_cast<float*>(smem + L::rr);
  float* cb_s = reinterpret_cast<float*>(smem + L::cb);
  uint64_t* full_x = reinterpret_cast<uint64_t*>(smem + L::bar);  // tile landed (TMA)
  uint64_t* bar_y = full_x + NX;    // rotation of a batch done
  uint64_t* bar_p = bar_y + NY;     // projection of a batch done
  uint64_t* yfree = bar_p + 2;      // Y of a batch read by the SIMT warps that take it (K: 16, V: 8)
  uint64_t* rready = yfree + NY;    // R of a batch stored by all 16 SIMT warps
  uint64_t* pfree = rready + 1;     // P of a batch read by all 16 SIMT warps
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::slot);
  const uint32_t sbase = tc::smem_addr(smem);

  if (warp == SIMT_WARPS) {
    tc::tmem_alloc(tmem_slot, kCols);
    if (lane == 0) {
      for (int i = 0; i < NX + NY + 2; ++i) tc::mbar_init(full_x + i, 1);
      for (int i = NX + NY + 2; i < L::n_bar; ++i) tc::mbar_init(full_x + i, QJL ? SIMT_WARPS : SIMT_WARPS / 2);
    }
  }
  if (threadIdx.x < 8) cb_s[threadIdx.x] = -a.tab.centroids[(B - 1) * 8 + threadIdx.x] * kRScale;  // -2^14 c
  if constexpr (QJL) {
    for (int i = threadIdx.x; i < 64 * 64; i += THREADS) {
      const int n = i >> 6, k = i & 63;
      const float hv = (__popc(n & k) & 1) ? -1.f : 1.f;
      const float ga = a.tab.signs[k] < 0 ? -hv : hv, gb = a.tab.signs[64 + k] < 0 ? -hv : hv;
      *reinterpret_cast<__half*>(smem + L::g + swz<64>(n, k)) = __float2half_rn(ga);
      *reinterpret_cast<__half*>(smem + L::g + kG + swz<64>(n, k)) = __float2half_rn(gb);
      *reinterpret_cast<__half*>(smem + L::g + 2 * kG + swz<64>(n, k)) = __float2half_rn(-gb);
    }
  } else {
    for (int i = threadIdx.x; i < D * D; i += THREADS) {  // (H D)[n][k] = (-1)^popcount(n & k) s_k
      const int n = i / D, k = i % D;
      const float hv = (__popc(n & k) & 1) ? -1.f : 1.f;
      *reinterpret_cast<__half*>(smem + L::g + swz<D>(n, k)) = __float2half_rn(a.tab.signs[k] < 0 ? -hv : hv);
    }
  }
  if constexpr (QJL) {
    for (int i = threadIdx.x; i < D * D; i += THREADS) {
      const int n = i / D, k = i % D;
      const float sv = a.tab.S[i];
      const __half hh = __float2half_rn(sv);
      *reinterpret_cast<__half*>(smem + L::s_hi + swz<128>(n, k)) = hh;
      *reinterpret_cast<__half*>(smem + L::s_lo + swz<128>(n, k)) = __float2half_rn(sv - __half2float(hh));
    }
  }
  tc::fence_async_smem();
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  const DevView& V = a.view;
  const long long nj = (sh.n_batches - blockIdx.x + gridDim.x - 1) / gridDim.x;  // batches of this CTA
  bool failed = false;

  if (issuer) {
    if (lane == 0) {
      // ---- issuers: tensor copies and MMAs, driven by the barriers ----
      long long next_tma = 0, mma1_done = 0, mma2_done = 0;  // counts issued
      auto issue_tma = [&](long long jj) {
        const uint32_t bt = (uint32_t)(blockIdx.x + jj * gridDim.x);
        const uint32_t l = fdiv(bt, sh.div_tb), tb = bt - l * sh.n_tb;
        uint64_t* fb = full_x + (int)(jj % NX);
        tc::mbar_arrive_expect_tx(fb, sh.tx_bytes);
        const uint32_t dst = sbase + L::x0 + (uint32_t)(jj % NX) * kOp;
        tc::tma_load_4d(dst, &tmap, 0, 0, (int)(tb * sh.TB), (int)l, fb);
        tc::tma_load_4d(dst + 128 * NV, &tmap, 64, 0, (int)(tb * sh.TB), (int)l, fb);
        next_tma = jj + 1;
      };
      // descriptors: the 14-bit start field (address / 16) of a base descriptor plus an offset
      const uint64_t dg = tc::desc_sw128(sbase + L::g);
      auto issue_mma1 = [&](long long jj) {
        const uint64_t dx = tc::desc_sw128(sbase + L::x0 + (uint32_t)(jj % NX) * kOp);
        const uint32_t d0 = tmem + (uint32_t)(jj % NY) * 128;
        if constexpr (QJL) {
          constexpr uint32_t id64 = tc::idesc_f16_f32(128, 64);
#pragma unroll
          for (int ks = 0; ks < 4; ++ks) {
            const uint64_t da = dx + (kstep<NV>(ks) >> 4), db = dx + (kstep<NV>(4 + ks) >> 4);
            const uint64_t go = kstep<64>(ks) >> 4;
            tc::mma_f16(d0, da, dg + go, id64, ks > 0);
            tc::mma_f16(d0, db, dg + (kG >> 4) + go, id64, true);
            tc::mma_f16(d0 + 64, da, dg + go, id64, ks > 0);
            tc::mma_f16(d0 + 64, db, dg + (2 * kG >> 4) + go, id64, true);
          }
        } else {
          constexpr uint32_t id128 = tc::idesc_f16_f32(128, 128);
#pragma unroll
          for (int ks = 0; ks < D / 16; ++ks)
            tc::mma_f16(d0, dx + (kstep<NV>(ks) >> 4), dg + (kstep<D>(ks) >> 4), id128, ks > 0);
        }
        tc::commit(bar_y + (int)(jj % NY));
        mma1_done = jj + 1;
      };
      auto issue_mma2 = [&](long long jj) {
        const uint64_t dh = tc::desc_sw128(sbase + L::x0 + (uint32_t)(jj % NX) * kOp);  // R_hi
        const uint64_t drl = tc::desc_sw128(sbase + L::r_lo);
        const uint64_t dsh = tc::desc_sw128(sbase + L::s_hi), dsl = tc::desc_sw128(sbase + L::s_lo);
        const uint32_t dp = tmem + 256 + (uint32_t)(jj & 1) * 128;
        constexpr uint32_t id128 = tc::idesc_f16_f32(128, 128);
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          const uint64_t ka = kstep<NV>(ks) >> 4, kb = kstep<D>(ks) >> 4;
          tc::mma_f16(dp, drl + ka, dsh + kb, id128, ks > 0);
          tc::mma_f16(dp, dh + ka, dsl + kb, id128, true);
          tc::mma_f16(dp, dh + ka, dsh + kb, id128, true);
        }
        tc::commit(bar_p + (jj & 1));
        mma2_done = jj + 1;
      };
      bool ok = true;
      if (warp == SIMT_WARPS) {
        // issuer A: tiles and rotations
        for (long long jj = 0; jj < NX && jj < nj; ++jj) issue_tma(jj);
        for (long long j = 0; ok && j <= nj; ++j) {
          // rotation of batch j: its tile landed, and Y[j % NY] (batch j - NY) was read
          if (j < nj) {
            ok = tc::mbar_wait(full_x + (int)(j % NX), (uint32_t)(j / NX) & 1u);
            if (ok && j >= NY) ok = tc::mbar_wait(yfree + (int)(j % NY), (uint32_t)((j - NY) / NY) & 1u);
            if (!ok) break;
            tc::fence_after_sync();
            issue_mma1(j);
          }
          // tile (j - 1) % NX is free once batch j - 1's last MMA (K: projection, V: rotation) completed
          const long long jp = j - 1;
          if (jp >= 0 && jp + NX < nj) {
            ok = QJL ? tc::mbar_wait(bar_p + (jp & 1), (uint32_t)(jp >> 1) & 1u)
                     : tc::mbar_wait(bar_y + (int)(jp % NY), (uint32_t)(jp / NY) & 1u);
            if (ok) issue_tma(jp + NX);
          }
        }
      } else {
        // issuer B (turbo K): projections, once R of the batch is stored and P[jp & 1] (batch jp - 2) was read
        for (long long jp = 0; ok && jp < nj; ++jp) {
          ok = tc::mbar_wait(rready, (uint32_t)jp & 1u);
          if (ok && jp >= 2) ok = tc::mbar_wait(pfree + (jp & 1), (uint32_t)((jp - 2) >> 1) & 1u);
          if (!ok) break;
          tc::fence_after_sync();
          issue_mma2(jp);
        }
      }
      if (!ok) {
        failed = true;
        // bounded waits for whatever this issuer still has in flight
        for (long long jj = mma1_done; jj < next_tma; ++jj)
          tc::mbar_wait(full_x + (int)(jj % NX), (uint32_t)(jj / NX) & 1u);
        if (mma1_done > 0) tc::mbar_wait(bar_y + (int)((mma1_done - 1) % NY), (uint32_t)((mma1_done - 1) / NY) & 1u);
        if (mma2_done > 0) tc::mbar_wait(bar_p + ((mma2_done - 1) & 1), (uint32_t)((mma2_done - 1) >> 1) & 1u);
      }
    }
  } else {
    // ---- SIMT warps ----
    float bnd[7];
#pragma unroll
    for (int k = 0; k < 7; ++k) bnd[k] = k < (1 << B) - 1 ? a.tab.boundaries[(B - 1) * 7 + k] : 0.f;
    float cst[7];
    const bool fma_idx = step_constants<B>(bnd, cst);  // the same on every thread
    constexpr int CPC = 8 * W <= 24 ? 8 : 4;           // codes per float-accumulated chunk
    const uint32_t lane_base = (uint32_t)(32 * q) << 16;
    uint32_t w_prev[W] = {};
    long long vid_prev = -1;
    float n_prev = 0.f;
    bool ok = true;
    if constexpr (!QJL) {
      // turbo-MSE V: two groups of 8 SIMT warps take alternate batches (group g the batches j with
      // j % 2 == g, in Y[j % 4]), so that one group's dependent steps overlap the other's; warp w of
      // a group reads lane quarter w % 4 and the column groups 2 hq, 2 hq + 1 (two passes of 32
      // columns, each read from tensor memory twice: for the norm, then for the codes), and the
      // group meets on its own named barrier (1 + g, 256 threads) for the norm exchange
      const int g = warp >> 3, hq = (warp >> 2) & 1;
      for (long long j = g; j < nj; j += 2) {
        const int yb = (int)(j % NY);
        ok = tc::mbar_wait(bar_y + yb, (uint32_t)(j / NY) & 1u) && ok;
        tc::fence_after_sync();
#pragma unroll
        for (int ps = 0; ps < 2; ++ps) {
          const int cgp = 2 * hq + ps;
          uint32_t t[32];
          tc::tmem_ld32(tmem + lane_base + yb * 128 + 32 * cgp, t);
          float2 ss2 = make_float2(0.f, 0.f);
#pragma unroll
          for (int e = 0; e < 32; e += 2) {
            const float2 yy = make_float2(__uint_as_float(t[e]), __uint_as_float(t[e + 1]));
            ss2 = __ffma2_rn(yy, yy, ss2);
          }
          ss_s[(yb * 4 + cgp) * NV + v] = ss2.x + ss2.y;
        }
        if (tc::bar_sync_or(1 + g, kSimt / 2, !ok)) {
          failed = true;
          break;
        }
        const uint32_t bt = (uint32_t)(blockIdx.x + j * gridDim.x);
        const uint32_t l = fdiv(bt, sh.div_tb), tb = bt - l * sh.n_tb;
        const int tok = (int)(tb * sh.TB) + tt;
        long long vid = -1;
        if (v < sh.rows && tok < a.n_tokens) vid = vid_at(a, (int)l, tok, h, hq == 0);
        const float* sp = ss_s + yb * 4 * NV + v;
        const float n = sqrtf((sp[0] + sp[NV] + sp[2 * NV] + sp[3 * NV]) * (1.f / D));  // |x| = |H D x| / sqrt(d)
        const float f = n > 0.f ? __fdividef(inv_sqrt_dim<D>(), n) : 0.f;
#pragma unroll
        for (int ps = 0; ps < 2; ++ps) {
          const int cgp = 2 * hq + ps;
          uint32_t t[32];
          tc::tmem_ld32(tmem + lane_base + yb * 128 + 32 * cgp, t);
          uint32_t w[W] = {};
          if (fma_idx) {
            const float F = f * 0x1p100f;
#pragma unroll
            for (int c = 0; c < 32 / CPC; ++c) {
              float2 acc2 = code_base<B, W, CPC>();
#pragma unroll
              for (int e = 0; e < CPC; e += 2) {
                const float2 cs = step_count_signed<B>(__uint_as_float(t[CPC * c + e]),
                                                       __uint_as_float(t[CPC * c + e + 1]), F, cst);
                acc2 = __ffma2_rn(cs, make_float2((float)(1u << (W * e)), (float)(1u << (W * (e + 1)))), acc2);
              }
              or_bits<W>(w, W * CPC * c, W * CPC, (uint32_t)(acc2.x + acc2.y));
            }
          } else {
#pragma unroll
            for (int e = 0; e < 32; ++e) put_code<W>(w, e, lloyd_index<B>(__uint_as_float(t[e]) * f, bnd));
          }
          if (vid >= 0) {
            if (cgp == 0) *reinterpret_cast<__half*>(V.header + vid * V.hdr_bytes) = __float2half_rn(n);
            store_words<W>(reinterpret_cast<uint32_t*>(V.payload + vid * V.pay_bytes) + W * cgp, w);
          }
        }
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(yfree + yb);
      }
    } else {
      for (long long j = 0; j < nj; ++j) {
        const int yb = (int)(j & 1);
        // (a) Y of batch j: partial sum of squares of this thread's 32 coordinates
        ok = tc::mbar_wait(bar_y + yb, (uint32_t)(j >> 1) & 1u) && ok;
        tc::fence_after_sync();
        uint32_t t[32];
        tc::tmem_ld32(tmem + lane_base + yb * 128 + 32 * cg, t);
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(yfree + yb);
        float2 ss2 = make_float2(0.f, 0.f);
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          const float2 yy = make_float2(__uint_as_float(t[e]), __uint_as_float(t[e + 1]));
          ss2 = __ffma2_rn(yy, yy, ss2);
        }
        const float ss = ss2.x + ss2.y;
        ss_s[(yb * 4 + cg) * NV + v] = ss;
        if (tc::bar_sync_or(1, kSimt, !ok)) {
          failed = true;
          break;
        }
        // (b) norm, destination
        const uint32_t bt = (uint32_t)(blockIdx.x + j * gridDim.x);
        const uint32_t l = fdiv(bt, sh.div_tb), tb = bt - l * sh.n_tb;
        const int tok = (int)(tb * sh.TB) + tt;
        long long vid = -1;
        if (v < sh.rows && tok < a.n_tokens) vid = vid_at(a, (int)l, tok, h, cg == 0);
        const float* sp = ss_s + yb * 4 * NV + v;
        const float n = sqrtf((sp[0] + sp[NV] + sp[2 * NV] + sp[3 * NV]) * (1.f / D));  // |x| = |H D x| / sqrt(d)
        const float f = n > 0.f ? __fdividef(inv_sqrt_dim<D>(), n) : 0.f;
        uint32_t w[W] = {};
        if constexpr (QJL) {
          // header of batch j - 1 (its residual partial sums were stored before the barrier)
          if (j > 0 && cg == 0 && vid_prev >= 0) {
            const float* rp = rr_s + (1 - yb) * 4 * NV + v;
            const float rs = (rp[0] + rp[NV] + rp[2 * NV] + rp[3 * NV]) * (1.f / (kRScale * kRScale));
            *reinterpret_cast<__half2*>(V.header + vid_prev * V.hdr_bytes) =
                __halves2half2(__float2half_rn(n_prev), __float2half_rn(n_prev * sqrtf(rs)));
          }
          // (c) index and residual; R_lo is free once the projection of batch j - 1 completed
          if (j > 0) {
            ok = tc::mbar_wait(bar_p + (1 - yb), (uint32_t)((j - 1) >> 1) & 1u) && ok;
            tc::fence_after_sync();
          }
          unsigned char* rh = smem + L::x0 + (int)(j % NX) * kOp;  // the rotation consumed X: R_hi goes there
          float2 rr2 = make_float2(0.f, 0.f);
          const float F = f * 0x1p100f, FR = f * kRScale;
          const uint32_t cbase = sbase + L::cb;
#pragma unroll
          for (int c8 = 0; c8 < 4; ++c8) {
            uint32_t hi[4], lo[4];
            if (fma_idx) {
              // pairs of coordinates in packed fp32 (even, odd): the code accumulators start at the
              // (H - 1/2) part of every index of their chunk, so the signed counts add the rest
              float2 acc2[8 / CPC];
#pragma unroll
              for (int c = 0; c < 8 / CPC; ++c) acc2[c] = code_base<B, W, CPC>();
#pragma unroll
              for (int e2 = 0; e2 < 8; e2 += 2) {
                const float ya = __uint_as_float(t[8 * c8 + e2]), yb = __uint_as_float(t[8 * c8 + e2 + 1]);
                const float2 cs = step_count_signed<B>(ya, yb, F, cst);
                // the index H - 1/2 + cs is an integer: as 2^21 + index it sits in bits 2..4, the byte
                // offset of its entry in the 32-byte-aligned table of -2^14 c
                constexpr float kIdx = (float)(1 << (B - 1)) - 0.5f + 0x1p21f;
                const float2 mg = __fadd2_rn(cs, make_float2(kIdx, kIdx));
                const float ca = lds_f32((__float_as_uint(mg.x) & 0x1Cu) | cbase);
                const float cb = lds_f32((__float_as_uint(mg.y) & 0x1Cu) | cbase);
                const float2 r2 = __ffma2_rn(make_float2(ya, yb), make_float2(FR, FR), make_float2(ca, cb));  // 2^14 (u - c)
                rr2 = __ffma2_rn(r2, r2, rr2);
                const int ep = e2 % CPC;
                acc2[e2 / CPC] = __ffma2_rn(cs, make_float2((float)(1u << (W * ep)), (float)(1u << (W * (ep + 1)))),
                                            acc2[e2 / CPC]);
                split_pair2(r2, hi[e2 / 2], lo[e2 / 2]);
              }
#pragma unroll
              for (int c = 0; c < 8 / CPC; ++c)
                or_bits<W>(w, W * (8 * c8 + CPC * c), W * CPC, (uint32_t)(acc2[c].x + acc2[c].y));
            } else {
#pragma unroll
              for (int e2 = 0; e2 < 8; e2 += 2) {
                const int e = 8 * c8 + e2;
                const float u0 = __uint_as_float(t[e]) * f, u1 = __uint_as_float(t[e + 1]) * f;
                const uint32_t i0 = lloyd_index<B>(u0, bnd), i1 = lloyd_index<B>(u1, bnd);
                const float r0 = fmaf(u0, kRScale, cb_s[i0]), r1 = fmaf(u1, kRScale, cb_s[i1]);  // 2^14 (u - c)
                rr2.x = fmaf(r0, r0, rr2.x);
                rr2.y = fmaf(r1, r1, rr2.y);
                put_code<W>(w, e, i0);
                put_code<W>(w, e + 1, i1);
                split_pair(make_float2(r0, r1), hi[e2 / 2], lo[e2 / 2]);
              }
            }
            const int off = swz<NV>(v, 32 * cg + 8 * c8);
            *reinterpret_cast<uint4*>(rh + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
            *reinterpret_cast<uint4*>(smem + L::r_lo + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
          }
          const float rr = rr2.x + rr2.y;
          rr_s[(yb * 4 + cg) * NV + v] = rr;
          tc::fence_async_smem();
          __syncwarp();
          if (lane == 0) tc::mbar_arrive(rready);
          // (e) sign bits of batch j - 1: its projection completed (waited above)
          if (j > 0) {
            uint32_t tp[32];
            tc::tmem_ld32(tmem + lane_base + 256 + (1 - yb) * 128 + 32 * cg, tp);
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(pfree + (1 - yb));
            uint32_t sbits = 0;
#pragma unroll
            for (int e = 0; e < 32; ++e) sbits |= (__uint_as_float(tp[e]) > 0.f ? 1u : 0u) << e;
            merge_signs<W, B>(w_prev, sbits);
            if (vid_prev >= 0)
              store_words<W>(reinterpret_cast<uint32_t*>(V.payload + vid_prev * V.pay_bytes) + W * cg, w_prev);
          }
#pragma unroll
          for (int k = 0; k < W; ++k) w_prev[k] = w[k];
          vid_prev = vid;
          n_prev = n;
        }
      }
    }
    if constexpr (QJL) {
      // the last batch: its header and sign bits
      if (!failed && tc::bar_sync_or(1, kSimt, !ok)) failed = true;
      if (!failed) {
        const long long jl = nj - 1;
        const int lb = (int)(jl & 1);
        if (cg == 0 && vid_prev >= 0) {
          const float* rp = rr_s + lb * 4 * NV + v;
          const float rs = (rp[0] + rp[NV] + rp[2 * NV] + rp[3 * NV]) * (1.f / (kRScale * kRScale));
          *reinterpret_cast<__half2*>(V.header + vid_prev * V.hdr_bytes) =
              __halves2half2(__float2half_rn(n_prev), __float2half_rn(n_prev * sqrtf(rs)));
        }
        if (tc::mbar_wait(bar_p + lb, (uint32_t)(jl >> 1) & 1u)) {
          tc::fence_after_sync();
          uint32_t tp[32];
          tc::tmem_ld32(tmem + lane_base + 256 + lb * 128 + 32 * cg, tp);
          uint32_t sbits = 0;
#pragma unroll
          for (int e = 0; e < 32; ++e) sbits |= (__uint_as_float(tp[e]) > 0.f ? 1u : 0u) << e;
          merge_signs<W, B>(w_prev, sbits);
          if (vid_prev >= 0)
            store_words<W>(reinterpret_cast<uint32_t*>(V.payload + vid_prev * V.pay_bytes) + W * cg, w_prev);
        } else {
          failed = true;
        }
      }
    }
  }
  if (failed) atomicOr(a.tab.status, kFlagTimeout);
  tc::fence_before_sync();
  __syncthreads();
  if (warp == SIMT_WARPS) tc::tmem_dealloc(tmem, kCols);
}

// cuTensorMapEncodeTiled from the driver (no link-time dependency on it); null if unavailable.
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static const PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      p = nullptr;
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }();
  return fn;
}

// Launches the tensor-core encoder; returns false (nothing launched) where its tensor map cannot
// describe the input, and the caller takes the register path.
template <bool QJL, int B>
bool launch_tc(const EncArgs& a, int sm_count, cudaStream_t s, cudaError_t* err) {
  using namespace etc;
  const int H = a.view.H;
  const auto encode = tensor_map_encoder();
  if (!encode || H > NV || a.n_tokens <= 0) return false;
  TcShape sh{};
  sh.H = H;
  sh.TB = NV / H;
  sh.rows = sh.H * sh.TB;
  sh.n_tb = (uint32_t)((a.n_tokens + sh.TB - 1) / sh.TB);
  sh.div_tb = make_fastdiv(sh.n_tb);
  sh.n_batches = (long long)a.n_layers * sh.n_tb;
  sh.tx_bytes = (uint32_t)(D / 8) * 8u * (uint32_t)sh.rows * 2u;
  if (sh.n_batches >= (1ll << 31)) return false;
  CUtensorMap tmap;
  const cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)a.n_tokens, (cuuint64_t)a.n_layers};
  const long long ts = a.token_stride * 2, ls = a.n_layers > 1 ? a.layer_stride * 2 : ts * a.n_tokens;
  if (ts <= 0 || ls <= 0) return false;
  const cuuint64_t strides[3] = {(cuuint64_t)D * 2, (cuuint64_t)ts, (cuuint64_t)ls};
  const cuuint32_t box[4] = {64, (cuuint32_t)H, (cuuint32_t)sh.TB, 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  if (encode(&tmap, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 4, const_cast<__half*>(a.x), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return false;
  constexpr size_t smem = Smem<QJL>::total + 1024;
  static_assert(smem <= 227 * 1024, "shared memory");
  auto kern = encode_tc_kernel<QJL, B>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e == cudaSuccess) {
    const long long grid = sh.n_batches < sm_count ? sh.n_batches : sm_count;  // one CTA per SM
    kern<<<(unsigned)grid, kThreads<QJL>, smem, s>>>(a, tmap, sh);
    e = cudaGetLastError();
  }
  *err = e;
  return true;
}

template <int D, bool QJL, int B>
cudaError_t launch_turbo(const EncArgs& a, int sm_count, cudaStream_t s) {
  using Sh = GroupShape<D>;
  constexpr int W = QJL ? B + 1 : B;
  size_t smem = 64;
  long long work;
  if (QJL) {
    smem += (size_t)Sh::NV * Sh::RS * 4 + (size_t)Sh::NV * Sh::L * W * 4 + (size_t)Sh::NV * (D / 32) * 4 +
            (size_t)Sh::NV * 8;
    work = (a.n_vectors + Sh::NV - 1) / Sh::NV;
  } else {
    work = (a.n_vectors + kEncWarps * Sh::VPW - 1) / (kEncWarps * Sh::VPW);
  }
  auto kern = encode_turbo_kernel<D, QJL, B>;
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

template <int D, bool QJL>
cudaError_t launch_turbo_bits(const EncArgs& a, int sm_count, cudaStream_t s) {
  if constexpr (D == 128) {
    cudaError_t e = cudaSuccess;
    bool done = false;
    switch (a.view.idx_bits) {
      case 1: done = launch_tc<QJL, 1>(a, sm_count, s, &e); break;
      case 2: done = launch_tc<QJL, 2>(a, sm_count, s, &e); break;
      case 3: done = launch_tc<QJL, 3>(a, sm_count, s, &e); break;
    }
    if (done) return e;
  }
  switch (a.view.idx_bits) {
    case 1: return launch_turbo<D, QJL, 1>(a, sm_count, s);
    case 2: return launch_turbo<D, QJL, 2>(a, sm_count, s);
    case 3: return launch_turbo<D, QJL, 3>(a, sm_count, s);
  }
  return cudaErrorInvalidValue;
}

template <int D, int KIND>
cudaError_t launch_kind(const EncArgs& a, int sm_count, cudaStream_t s) {
  const size_t smem = (size_t)kEncWarps * D;
  const long long work = (a.n_vectors + 8 * kEncWarps - 1) / (8 * kEncWarps);  // runs of 8 vectors per warp
  auto kern = encode_kernel<D, KIND>;
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
  if (a.view.has_qjl) return launch_turbo_bits<D, true>(a, sm_count, s);
  return launch_turbo_bits<D, false>(a, sm_count, s);
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
