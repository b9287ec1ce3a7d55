// Split-K decode attention on tensor cores for turbo4 K (3-bit index + QJL
// sign per coordinate, stored as nibbles) and turbo4_mse V (3-bit index),
// head_dim 128, up to 4 query heads per KV head (5 to 8 take the
// format-parameterised kernel of tq_decode_mma.cuh, whose two products per part
// keep the query columns split into high and low parts).  Same contract as the
// generic kernel in tq_decode.cu: one partial (m, l, acc) per (query row,
// split), combined afterwards.
//
// Per warp, tiles of 16 tokens:
//   * scores on mma.sync m16n8k16 (f16 in, f32 accumulate), two products per
//     tile and k step, rows = the 16 tokens: one of the codebook parts c[idx]
//     against q', one of the QJL parts (2 sigma - 1) against S q'.  Both parts
//     of two coordinates of one token come from one 8-byte lookup, indexed by
//     one payload byte (index + sign nibbles), in a 256-entry table in shared
//     memory: its first word goes to the codebook product's A fragment, its
//     second to the QJL product's.  The contraction index is permuted so that
//     thread t's k slots are coordinates of its own 32-coordinate block of
//     tokens g and g + 8 (the query fragments follow the same permutation), so
//     four lookups fill the two A fragments as they stand and every output of
//     both products is used.  The table is replicated per lane (entry stride
//     256 B, lane offset 8 B) so the 32 lookups of a warp never collide, and
//     it starts on a 64 KB boundary of the shared window, so one prmt of the
//     payload word with (table base | lane << 3) is the whole address.
//     score = n * (c . q') + rnorm * (sign . S q') (per token; 1/lambda,
//     log2 e and sqrt(pi/2)/d are folded into the query columns).
//   * online softmax in registers (base 2), with a lazily raised reference:
//     only when a score passes it by 2^8 are the sums and accumulators rescaled;
//   * Sparse V: a tile whose every weight is below the threshold skips V,
//     inside a kept tile weights below it are zeroed;
//   * O^T[128 dims x 8 cols] += V~^T . P' on mma.sync m16n8k16 (f16 in, f32
//     accumulate), P' = weight * V norm.  A 64-entry table (8 KB aligned, so
//     one shift and one lop3 form the address) indexed by the 6-bit code of
//     two coordinates of one token returns their f16 pair; one prmt per
//     register then pairs two tokens at the same coordinate, which is the
//     fragment layout of a contraction over tokens.  The k slots of that
//     contraction hold the tokens in the order 0, 8, 1, 9, ..., so each thread
//     stores its two tokens' weights of one column as one 32-bit word.
// Query heads: the 8 columns of a score product.  Column 2h holds the high and
// column 2h + 1 the low fp16 part of head h's q' (or S q'), about 21
// significant bits, and in the V product column 2t holds head t's weights as
// the high part and column 2t + 1 as the low part; thread (g, t) owns head t.
//
// The fp16 tables hold lambda * centroid, lambda chosen on the host so that
// every entry is within ~2e-5 of its fp32 value; 1/lambda goes into the query
// columns (K) and into the partial's accumulator (V).
//
// Work: a work item is (layer x sequence, KV head, split of the context); each
// warp takes items from an atomic counter (zeroed by the prologue kernel) and
// writes one partial per query head and item, so warps never wait for each
// other.  Memory: the K and V bytes of the tiles 4 and 5 ahead are requested
// into L2 with bulk prefetches every second tile, so a tile's own register loads
// (K at its start, V after the K contraction) meet L2 and registers hold one
// tile only; cache loads carry an evict-first L2 policy so that the partials
// stay in L2 for the combine.
// One persistent CTA of 16 warps per SM.
#include <cuda_fp16.h>

#include "tq_device.cuh"
#include "tq_warp_mma.cuh"

namespace tq {
namespace {

using namespace wm;

constexpr int kFD = 128;
constexpr int kFWarps = 16;
constexpr int kFThreads = kFWarps * 32;

constexpr uint32_t kLutKBytes = 256 * 256;        // 256 entries x 32 lanes x 8 B
constexpr uint32_t kLutVBytes = 64 * 128;         // 64 entries x 32 lanes x 4 B
constexpr uint32_t kPsBytes = kFWarps * 2 * 256;  // per warp two P' tiles [8 cols][16 tokens] f16
constexpr int kQfBytes = 32 * 32 * 4;             // per warp: the query fragments, 32 words x 32 lanes
// The K table on a 64 KB boundary, the V table and the P' tiles next to it all end below 128 KB
// (the table starts below 64 KB, and the other two fit on one side of it); the query fragments
// of the warps follow at 128 KB.
constexpr int kFSmem = 2 * 65536 + kFWarps * kQfBytes;
constexpr int kPrefetchTiles = 4;                 // L2 prefetch distance

// Bytes per token of the two formats (d = 128).
constexpr int kKPay = 64, kKHdr = 4, kVPay = 48, kVHdr = 2;

// Address of the K table entry for byte kk of word x: table base | x.byte[kk] << 8 | lane << 3.
template <int KK>
__device__ __forceinline__ uint32_t lutk_addr(uint32_t x, uint32_t ylk) {
  return __byte_perm(x, ylk, 0x7604 | (KK << 4));
}

// Address of the V table entry for the 6-bit code at bit S of w: table base | code << 7 | lane << 2.
template <int S>
__device__ __forceinline__ uint32_t lutv_addr(uint32_t w, uint32_t ylv) {
  const uint32_t x = S >= 7 ? (w >> (S - 7)) : (w << (7 - S));
  return (x & 0x1F80u) | ylv;
}

struct KTile {
  uint4 a, b;       // payload block t of tokens g, g + 8
  uint32_t ha, hb;  // headers (fp16 n, fp16 rnorm) of tokens g, g + 8
};
struct VTile {
  uint32_t w[4][2];  // code words of tokens t, t + 8, t + 4, t + 12
  uint32_t nv;       // fp16 norms of tokens g (low) and g + 8 (high)
};

// Cache position of a warp's current tile and its lanes' load addresses.
struct Cursor {
  const unsigned char *kp, *kh, *vp, *vh;  // this lane's addresses in the current tile
  int in_page, page_ord;                   // token offset in its page; logical page
  bool ok;                                 // page in range
};

// Columns 2h and 2h + 1 of the score products and of P' hold the high and the low fp16 parts of
// query head h (up to 4 heads per KV head); thread (g, t) owns head t.
struct FastWarp {

  const DecodeLaunch& k;
  int lane, g, t;
  uint32_t ylk, ylv;         // table bases | lane offsets
  uint32_t psw0, psw1, psr;  // shared addresses of this lane's P' words in the warp's first P' tile
  uint32_t vsh;              // bit offset of coordinate 16g's V code in its word
  uint64_t pol;              // evict-first L2 policy

  // per work item
  int layer, b, kvh, ntiles, last_valid;
  Cursor c;
  uint32_t qf;  // shared address of this lane's query fragments: step ch at qf + 256 ch (codebook
                // product), qf + 2048 + 256 ch (QJL product), 8 bytes each
  float oacc[8][4];
  float m, l;  // running reference and sum of head t

  __device__ __forceinline__ FastWarp(const DecodeLaunch& k_) : k(k_) {}

  __device__ __forceinline__ void set_page() {
    const DecodeArgs& a = k.a;
    long long page = b;
    c.ok = true;
    if (a.block_table) {
      page = a.block_table[(long long)b * a.max_blocks_per_seq + c.page_ord];
      if (page < 0 || page >= a.k.num_pages) {
        if (lane == 0) atomicOr(k.tab.status, kFlagBlockTable);
        c.ok = false;
        page = 0;
      }
    }
    const long long base = (((long long)layer * a.k.num_pages + page) * a.k.H + kvh) * a.k.page_size + c.in_page;
    c.kp = a.k.payload + (base + g) * kKPay + 16 * t;
    c.kh = a.k.header + (base + g) * kKHdr;
    c.vp = a.v.payload + (base + t) * kVPay + 4 * ((3 * g) >> 1);
    c.vh = a.v.header + (base + g) * kVHdr;
  }

  __device__ __forceinline__ void advance() {
    c.in_page += 16;
    if (c.in_page == k.a.k.page_size) {
      c.in_page = 0;
      ++c.page_ord;
      set_page();
    } else {
      c.kp += 16 * kKPay;
      c.kh += 16 * kKHdr;
      c.vp += 16 * kVPay;
      c.vh += 16 * kVHdr;
    }
  }

  // K of a tile whose lane addresses are kp, kh (this lane's rows g, g + 8)
  __device__ __forceinline__ void load_k(KTile& K, const unsigned char* kp, const unsigned char* kh, int nvalid) {
    if (nvalid == 16) {
      K.a = ld_stream_v4(kp, pol);
      K.b = ld_stream_v4(kp + 8 * kKPay, pol);
      K.ha = ld_stream_u32(kh, pol);
      K.hb = ld_stream_u32(kh + 8 * kKHdr, pol);
    } else {  // ragged last tile: rows at or beyond nvalid re-read row nvalid - 1 (their scores are masked)
      const int da = min(g, nvalid - 1) - g, db = min(g + 8, nvalid - 1) - g;
      K.a = ld_stream_v4(kp + da * kKPay, pol);
      K.b = ld_stream_v4(kp + db * kKPay, pol);
      K.ha = ld_stream_u32(kh + da * kKHdr, pol);
      K.hb = ld_stream_u32(kh + db * kKHdr, pol);
    }
  }

  __device__ __forceinline__ void load_v(VTile& V, int nvalid) {
    if (nvalid == 16) {
      const int off[4] = {0, 8 * kVPay, 4 * kVPay, 12 * kVPay};
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        V.w[r][0] = ld_stream_u32(c.vp + off[r], pol);
        V.w[r][1] = ld_stream_u32(c.vp + off[r] + 4, pol);
      }
      V.nv = ld_stream_u16(c.vh, pol) | (ld_stream_u16(c.vh + 8 * kVHdr, pol) << 16);
    } else {
      const int rows[4] = {t, t + 8, t + 4, t + 12};
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const unsigned char* p = c.vp + (min(rows[r], nvalid - 1) - t) * kVPay;
        V.w[r][0] = ld_stream_u32(p, pol);
        V.w[r][1] = ld_stream_u32(p + 4, pol);
      }
      V.nv = ld_stream_u16(c.vh + (min(g, nvalid - 1) - g) * kVHdr, pol) |
             (ld_stream_u16(c.vh + (min(g + 8, nvalid - 1) - g) * kVHdr, pol) << 16);
    }
  }

  // Header tiles start on 16-byte boundaries (bulk prefetch) when pages hold a multiple of
  // 16 tokens and both header arrays are 16-byte aligned.
  __device__ __forceinline__ bool headers_aligned() const {
    return k.a.k.page_size % 16 == 0 &&
           ((reinterpret_cast<uintptr_t>(k.a.k.header) | reinterpret_cast<uintptr_t>(k.a.v.header)) & 15) == 0;
  }

  // Requests tiles [tile + ahead, tile + ahead + n) into L2, n <= count, clipped to the work
  // item and to the page (lane 0, whose addresses are the current tile's own).
  __device__ __forceinline__ void prefetch_tiles(int tile, int ahead, int count) {
    const int n = min(min(ntiles - tile - ahead, count), (k.a.k.page_size - c.in_page) / 16 - ahead);
    if (lane != 0 || n <= 0 || !c.ok) return;
    prefetch_l2(c.kp + 16 * ahead * kKPay, 16 * n * kKPay);
    prefetch_l2(c.vp + 16 * ahead * kVPay, 16 * n * kVPay);
    if (headers_aligned()) {
      prefetch_l2(c.kh + 16 * ahead * kKHdr, 16 * n * kKHdr);
      prefetch_l2(c.vh + 16 * ahead * kVHdr, 16 * n * kVHdr);
    }
  }

  // Raises the reference of every head whose new scores pass it by 2^8 (warp-uniform decision).
  __device__ __forceinline__ void raise_reference(float mx) {
    if (!__any_sync(kFull, mx > m + kLazyMax)) return;
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, o));
    const float mn = fmaxf(m, mx);
    const float al = ex2(m - mn);
    l *= al;
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) {
#pragma unroll
      for (int e = 0; e < 4; ++e) oacc[mt][e] *= al;
    }
    m = mn;
  }

  // One tile at the cursor (the caller advances the cursor afterwards).
  template <int BUF>
  __device__ __forceinline__ void step(int tile) {
    const int nvalid = tile == ntiles - 1 ? last_valid : 16;
    if (!c.ok) {  // warp-uniform: the tile's page was out of range
      __syncwarp();
      return;
    }
    KTile kc;
    load_k(kc, c.kp, c.kh, nvalid);

    // ---- K: rows = tokens g / g + 8 of the thread; cc = codebook part . q', cs = QJL part . S q' ----
    float cc[4] = {0.f, 0.f, 0.f, 0.f}, cs[4] = {0.f, 0.f, 0.f, 0.f};
    const uint32_t wa[4] = {kc.a.x, kc.a.y, kc.a.z, kc.a.w};
    const uint32_t wb[4] = {kc.b.x, kc.b.y, kc.b.z, kc.b.w};
#pragma unroll
    for (int ch = 0; ch < 8; ++ch) {
      const uint32_t xa = wa[ch >> 1], xb = wb[ch >> 1];
      uint2 ea0, ea1, eb0, eb1;
      if (ch & 1) {
        ea0 = lds64(lutk_addr<2>(xa, ylk)); ea1 = lds64(lutk_addr<3>(xa, ylk));
        eb0 = lds64(lutk_addr<2>(xb, ylk)); eb1 = lds64(lutk_addr<3>(xb, ylk));
      } else {
        ea0 = lds64(lutk_addr<0>(xa, ylk)); ea1 = lds64(lutk_addr<1>(xa, ylk));
        eb0 = lds64(lutk_addr<0>(xb, ylk)); eb1 = lds64(lutk_addr<1>(xb, ylk));
      }
      const uint2 fq = lds64(qf + 256 * ch), fs = lds64(qf + 2048 + 256 * ch);
      mma_16816(cc, ea0.x, eb0.x, ea1.x, eb1.x, fq.x, fq.y);
      mma_16816(cs, ea0.y, eb0.y, ea1.y, eb1.y, fs.x, fs.y);
    }
    VTile vc;
    load_v(vc, nvalid);
    // thread (g, t): entries 0, 1 = token g, columns 2t, 2t + 1 (the two parts of head t);
    // entries 2, 3 = token g + 8.
    const float2 hA = __half22float2(u32_as_h2(kc.ha)), hB = __half22float2(u32_as_h2(kc.hb));
    float s0 = fmaf(hA.x, cc[0] + cc[1], hA.y * (cs[0] + cs[1]));
    float s1 = fmaf(hB.x, cc[2] + cc[3], hB.y * (cs[2] + cs[3]));
    if (nvalid < 16) {
      if (g >= nvalid) s0 = -INFINITY;
      if (g + 8 >= nvalid) s1 = -INFINITY;
    }

    // ---- online softmax with a lazily raised reference (base 2) ----
    raise_reference(fmaxf(s0, s1));
    float p0 = ex2(s0 - m), p1 = ex2(s1 - m);
    l += p0 + p1;
    // ---- Sparse V: weights below the threshold are dropped; an all-dropped tile skips V ----
    if (k.a.skip_threshold > 0.f) {
      const float tau = k.a.skip_threshold;
      p0 = p0 >= tau ? p0 : 0.f;
      p1 = p1 >= tau ? p1 : 0.f;
      if (!__any_sync(kFull, (p0 + p1) > 0.f)) {
        __syncwarp();
        return;
      }
    }

    // ---- P' = weight * V norm, one word per (column, token pair g / g + 8) ----
    const float2 nv = __half22float2(u32_as_h2(vc.nv));
    constexpr uint32_t kBuf = 256 * BUF;
    {
      const float w0 = p0 * nv.x, w1 = p1 * nv.y;
      const __half2 hi = __floats2half2_rn(w0, w1);
      const float2 hf = __half22float2(hi);
      sts32(psw0 + kBuf, h2_as_u32(hi));
      sts32(psw1 + kBuf, h2_as_u32(__floats2half2_rn(w0 - hf.x, w1 - hf.y)));
    }
    __syncwarp();
    const uint2 bp = lds64_v(psr + kBuf);

    // ---- V: O^T[16 dims x 8 cols] += V~^T[16 dims x 16 token slots] . P'[16 slots x 8 cols] ----
    // rows g / g + 8 of m-tile mt = coordinates 16g + 2mt / + 1
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
        uint32_t ad;
        switch (mt) {
          case 0: ad = lutv_addr<0>(xl[r], ylv); break;
          case 1: ad = lutv_addr<6>(xl[r], ylv); break;
          case 2: ad = lutv_addr<12>(xl[r], ylv); break;
          case 3: ad = lutv_addr<18>(xl[r], ylv); break;
          case 4: ad = lutv_addr<24>(xl[r], ylv); break;
          case 5: ad = lutv_addr<7>(__funnelshift_r(xl[r], xh[r], 23), ylv); break;
          case 6: ad = lutv_addr<4>(xh[r], ylv); break;
          default: ad = lutv_addr<10>(xh[r], ylv); break;
        }
        e[r] = lds32(ad);  // (c[2p], c[2p+1]) of one token
      }
      // a0/a1: slots 2t, 2t+1 = tokens t, t+8 at coordinate 2p / 2p+1; a2/a3: tokens t+4, t+12
      mma_16816(oacc[mt], __byte_perm(e[0], e[1], 0x5410), __byte_perm(e[0], e[1], 0x7632),
                __byte_perm(e[2], e[3], 0x5410), __byte_perm(e[2], e[3], 0x7632), bp.x, bp.y);
    }
  }

  __device__ __forceinline__ void run_item(unsigned int item) {
    const DecodeArgs& a = k.a;
    const int H = a.k.H, G = k.G, Hq = a.n_q_heads;
    const int split = (int)(item % k.n_splits);
    const unsigned int rest = item / k.n_splits;
    kvh = (int)(rest % H);
    const int lb = (int)(rest / H);
    layer = a.layer_begin + lb / a.batch;
    b = lb % a.batch;
    int len = a.seq_lens[b];
    if (len < 0) len = 0;
    if (len > a.max_ctx) {
      if (lane == 0) atomicOr(k.tab.status, kFlagSeqLen);
      len = a.max_ctx;
    }
    const int t0 = split * k.split_tokens;
    const int t1 = min(t0 + k.split_tokens, len);
    const long long row0 = (long long)lb * Hq + (long long)kvh * G;

    // ---- B fragments, column g: head g/2, the high (g even) or low (g odd) fp16 part.
    // Codebook product: q' with log2 e / lambda folded in; QJL
    // product: S q' with log2 e sqrt(pi/2) / d.  k slots 2t, 2t + 1 (+8) of step ch = coordinates
    // 32t + 4ch + {0, 1} ({2, 3}), as the A fragments have them ----
    {
      const int head = g >> 1;
      const bool lo = g & 1;
      const bool valid = head < G;
      const float* qp = k.qprep + (row0 + (valid ? head : 0)) * 2 * kFD + 32 * t;
      const float fq = valid ? kLog2e / k.tab.f16_scale[2] : 0.f;
      const float fs = valid ? kLog2e * kSqrtHalfPi / (float)kFD : 0.f;
#pragma unroll
      for (int ch = 0; ch < 8; ++ch) {
        const float4 v = *reinterpret_cast<const float4*>(qp + 4 * ch);
        const float4 u = *reinterpret_cast<const float4*>(qp + kFD + 4 * ch);
        sts64(qf + 256 * ch, pack_part(v.x * fq, v.y * fq, lo), pack_part(v.z * fq, v.w * fq, lo));
        sts64(qf + 2048 + 256 * ch, pack_part(u.x * fs, u.y * fs, lo), pack_part(u.z * fs, u.w * fs, lo));
      }
      __syncwarp();  // the lanes' own fragments only, but keep the stores ahead of the first read
    }
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) oacc[mt][0] = oacc[mt][1] = oacc[mt][2] = oacc[mt][3] = 0.f;
    m = -INFINITY;
    l = 0.f;

    ntiles = t1 > t0 ? (t1 - t0 + 15) / 16 : 0;
    last_valid = t1 - t0 - 16 * (ntiles - 1);
    if (ntiles > 0) {
      c.page_ord = t0 / a.k.page_size;
      c.in_page = t0 - c.page_ord * a.k.page_size;
      set_page();
      prefetch_tiles(0, 0, kPrefetchTiles);
      for (int tile = 0; tile < ntiles; tile += 2) {
        prefetch_tiles(tile, kPrefetchTiles, 2);  // the two tiles that follow the ones already requested
        step<0>(tile);
        if (tile + 1 >= ntiles) break;
        advance();
        step<1>(tile + 1);
        if (tile + 2 >= ntiles) break;
        advance();
      }
    }

    // ---- partial of this work item: (m, l, acc) of head t ----
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) l += __shfl_xor_sync(kFull, l, o);
    if (t < G) {
      const float inv_lam = 1.0f / k.tab.f16_scale[2];
      float v[16];
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) {
        v[2 * mt] = (oacc[mt][0] + oacc[mt][1]) * inv_lam;
        v[2 * mt + 1] = (oacc[mt][2] + oacc[mt][3]) * inv_lam;
      }
      float* dst = k.partial + ((row0 + t) * k.n_splits + split) * (kFD + 4);
      float4* dv = reinterpret_cast<float4*>(dst + 4 + 16 * g);
#pragma unroll
      for (int q = 0; q < 4; ++q) dv[q] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
      if (g == 0) {
        dst[0] = m == -INFINITY ? -INFINITY : m * kLn2;
        dst[1] = l;
      }
    }
  }

  // Two f16 B-fragment halves: the high (or low) fp16 part of x0, x1.
  static __device__ __forceinline__ uint32_t pack_part(float x0, float x1, bool lo) {
    const __half2 hi = __floats2half2_rn(x0, x1);
    if (!lo) return h2_as_u32(hi);
    const float2 hf = __half22float2(hi);
    return h2_as_u32(__floats2half2_rn(x0 - hf.x, x1 - hf.y));
  }
};

__global__ void __launch_bounds__(kFThreads, 1) attend_fast_kernel(DecodeLaunch k) {
  extern __shared__ __align__(16) unsigned char sm[];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  // ---- shared layout: K table on a 64 KB boundary of the shared window, V table on 8 KB ----
  const uint32_t sbase = static_cast<uint32_t>(__cvta_generic_to_shared(sm));
  const uint32_t kofs = (0x10000u - (sbase & 0xFFFFu)) & 0xFFFFu;
  uint32_t vofs, pofs;
  if (kofs >= kLutVBytes + kPsBytes) {
    vofs = kofs - kLutVBytes;
    pofs = vofs - kPsBytes;
  } else {
    vofs = kofs + kLutKBytes;
    pofs = vofs + kLutVBytes;
  }
  {
    const float* cb = k.tab.centroids + 2 * 8;  // 3-bit codebook
    const float lam = k.tab.f16_scale[2];
    for (int i = tid; i < 256 * 32; i += kFThreads) {
      const int e = i >> 5, r = i & 31, lo = e & 15, hi = e >> 4;
      uint2 v;
      v.x = h2_as_u32(__floats2half2_rn(lam * cb[lo & 7], lam * cb[hi & 7]));
      v.y = h2_as_u32(__floats2half2_rn((lo >> 3) ? 1.f : -1.f, (hi >> 3) ? 1.f : -1.f));
      *reinterpret_cast<uint2*>(sm + kofs + e * 256 + r * 8) = v;
    }
    for (int i = tid; i < 64 * 32; i += kFThreads) {
      const int e = i >> 5, r = i & 31;
      *reinterpret_cast<uint32_t*>(sm + vofs + e * 128 + r * 4) =
          h2_as_u32(__floats2half2_rn(lam * cb[e & 7], lam * cb[e >> 3]));
    }
  }
  __syncthreads();

  FastWarp w(k);
  w.lane = lane;
  w.g = lane >> 2;
  w.t = lane & 3;
  w.ylk = (sbase + kofs) | ((uint32_t)lane << 3);
  w.ylv = (sbase + vofs) | ((uint32_t)lane << 2);
  const uint32_t ps = sbase + pofs + warp * 512;  // this warp's two P' tiles of 64 words
  w.psw0 = ps + 4 * ps_word(2 * w.t, w.g);
  w.psw1 = ps + 4 * ps_word(2 * w.t + 1, w.g);
  w.psr = ps + 4 * ps_word(w.g, w.t);
  w.vsh = (w.g & 1) ? 16u : 0u;
  w.qf = sbase + 2 * 65536 + warp * (uint32_t)kQfBytes + lane * 8;
  asm("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(w.pol));

  const DecodeArgs& a = k.a;
  const unsigned int n_items = (unsigned int)((long long)a.n_layers * a.batch * a.k.H * k.n_splits);
  for (;;) {
    unsigned int item = 0;
    if (lane == 0) item = atomicAdd(k.counter, 1u);
    item = __shfl_sync(kFull, item, 0);
    if (item >= n_items) break;
    __syncwarp();  // the previous item's P' reads are done before this item's writes
    w.run_item(item);
  }
}

}  // namespace

bool attend_fast_supported(const DecodeLaunch& k) {
  const DecodeArgs& a = k.a;
  return a.k.d == kFD && a.k.format == TQ_FMT_TURBO4 && a.v.format == TQ_FMT_TURBO4_MSE && k.G >= 1 &&
         k.G <= 4 && (a.block_table == nullptr || a.k.page_size % 16 == 0) && k.split_tokens % 16 == 0;
}

cudaError_t launch_attend_fast(const DecodeLaunch& k, int sm_count, cudaStream_t s) {
  const long long items = (long long)k.a.n_layers * k.a.batch * k.a.k.H * k.n_splits;
  if (items >= (1LL << 32)) return cudaErrorInvalidValue;
  long long grid = sm_count;  // one persistent CTA per SM
  if (items < grid * kFWarps) grid = (items + kFWarps - 1) / kFWarps;
  if (grid < 1) grid = 1;
  const cudaError_t e = cudaFuncSetAttribute(attend_fast_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kFSmem);
  if (e != cudaSuccess) return e;
  attend_fast_kernel<<<(unsigned)grid, kFThreads, kFSmem, s>>>(k);
  return cudaGetLastError();
}

}  // namespace tq
