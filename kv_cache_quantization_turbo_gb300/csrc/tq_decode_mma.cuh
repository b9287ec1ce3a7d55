// Split-K decode attention on tensor cores, parameterised by the cache formats: turbo K with
// W-bit codes (W - 1 index bits + the QJL sign bit; turbo2/3/4), turbo-MSE V with W-bit indices
// (turbo2/3/4_mse), and q8_0 K or V, at head_dim 64, 128 or 256, up to 16 query heads per KV head
// per work item at d <= 128 (up to 8 at d = 256: with 9 to 16 every item runs twice there, on the
// two halves of the heads, as consecutive work-counter values).  One partial (m, l, acc) per query
// row and split, combined afterwards.
//
// Why tensor cores: at HBM speed one 16-token tile of one KV head (1888 B for turbo4 / turbo4_mse
// at d = 128) leaves ~350 warp instructions per SM, and scoring it on CUDA cores takes ~3 G d
// FMAs per token; the contraction over the G query heads of a KV head is a dense (16 tokens x d)
// x (d x G) product per tile, so it and the V accumulation run on mma.sync m16n8k16 (f16 in, f32
// accumulate) over operands dequantised by table lookups.
//
// Work: a work item is (layer x sequence, KV head, split of the context); each warp takes items
// from an atomic counter (zeroed by the prologue kernel) and writes one partial per query head
// and item, so warps never wait for each other.  One persistent CTA per SM.  Per tile of 16
// tokens: K loads, score products, online softmax in registers (base 2, with a reference raised
// lazily: only when a score passes it by 2^8 are the sums and accumulators rescaled), Sparse V
// (a tile whose every weight is below the threshold skips V; inside a kept tile weights below it
// are zeroed), P' into a per-warp shared tile, V loads, V products.  Memory: every second tile one
// lane requests the two tiles 3-4 ahead into L2 (cp.async.bulk.prefetch; contiguous caches: the
// tiles of a page), so a tile's own register loads meet L2; cache loads carry an evict-first L2
// policy so that the partials stay in L2 for the combine.
//
// Tables: entries replicated per lane (lane offset 8 or 4 bytes, entry stride 256 or 128 bytes)
// so a warp's 32 lookups never collide, each table on a boundary of its own size so that the
// address is the code bits shifted into place OR (table base | lane offset).  They hold
// lambda * centroid in fp16, lambda chosen on the host so that every entry is within ~2e-5 of
// its fp32 value; 1/lambda goes into the query columns (K) and the partial's accumulator (V).
//
// Score products (mma.sync m16n8k16, rows = the 16 tokens of a tile, columns 2h / 2h + 1 = the
// high / low fp16 part of query head h, about 21 significant bits of q'; with 5 to 8 query heads
// per KV head a second product of each kind takes heads 4 .. 7).  Thread (g, t) holds rows g,
// g + 8, the scores of heads t (and t + 4), and per k step the four k slots 2t, 2t + 1, 2t + 8,
// 2t + 9:
//   * turbo K: thread t owns the coordinates [t d/4, (t+1) d/4) of its tokens, a contiguous run
//     of d W / 4 payload bits; step ch takes coordinates 4ch .. 4ch + 3 of the run.  The 2W bits
//     of two coordinates index a table of 8-byte entries (replicated per lane, entry stride
//     256 B): the f16 pair lambda c[idx] for the codebook product (against q') and the pair of
//     +-1 for the QJL product (against S q').  score = n (c . q') + rnorm sqrt(pi/2)/d (sign . Sq').
//   * q8_0 K: step ch covers 16 coordinates of the 32-block ch / 2, thread t holding bytes
//     8t + 4 (ch & 1) .. + 3 of the block; signed bytes become exact f16 pairs, the block's two
//     steps accumulate into fresh registers, and the block's fp16 scale multiplies that sum in
//     fp32.  score = sum over blocks of delta_b (int8_b . q'_b).
// V product: O^T[d x 8 columns] += V~^T[d x 16 token slots] . P'[16 slots x 8 columns], thread
// (g, t) holding rows g, g + 8 of m tile mt = coordinates g d/8 + 2mt, + 1, and token slots
// t, t + 8 (fragment registers 0, 1) and t + 4, t + 12 (registers 2, 3):
//   * turbo-MSE V: the 2W bits of two coordinates index a table of f16 pairs lambda c[idx]
//     (entry stride 128 B); the V norm goes into P' = weight * norm;
//   * q8_0 V: the signed bytes of two tokens at one coordinate become an f16 pair, multiplied by
//     the two tokens' block scales (f16); P' = weight.
// The V product's k slots hold the tokens in the order 0, 8, 1, 9, ..., so one byte permute per
// register pairs two tokens' table entries at one coordinate (the fragment layout of a contraction
// over tokens), and each thread stores its two tokens' weights of one column as one 32-bit word.
// P' columns: up to 4 heads, 2t / 2t + 1 = high / low fp16 part of head t's P'; 5 to 8 heads,
// heads t and t + 4 in plain fp16 (a relative rounding of 2^-12 per weight; the query side needs
// the split, since a score's rounding error grows with the score).
#pragma once

#include <cuda_fp16.h>

#include "tq_device.cuh"
#include "tq_warp_mma.cuh"

namespace tq {
namespace mmad {

using namespace wm;

constexpr int kPrefetchTiles = 3;  // L2 prefetch distance in tiles

// Most 32-bit words that cover bits [s, s + n) for the starts s = i n, i < count.
constexpr int cover_words(int n, int count) {
  int m = 0;
  for (int i = 0; i < count; ++i) {
    const int w = ((i * n) % 32 + n + 31) / 32;
    m = w > m ? w : m;
  }
  return m;
}
// Largest of 16, 8, 4 that divides both a and b.
constexpr int vec_bytes(int a, int b) { return (a % 16 == 0 && b % 16 == 0) ? 16 : (a % 8 == 0 && b % 8 == 0) ? 8 : 4; }

// Shape of one kernel: head_dim D, K code width WK (0 = q8_0), V code width WV (0 = q8_0).
template <int D_, int WK_, int WV_>
struct Fmt {
  static constexpr int D = D_, WK = WK_, WV = WV_;
  static constexpr bool KQ8 = WK == 0, VQ8 = WV == 0;
  static constexpr int KS = D / 16;  // k steps of a score product = m tiles of the V product
  static constexpr int KPay = KQ8 ? D : D * WK / 8, KHdr = KQ8 ? D / 16 : 4;
  static constexpr int VPay = VQ8 ? D : D * WV / 8, VHdr = VQ8 ? D / 16 : 2;
  // K words per thread and token.  turbo: the d W / 4-bit run at bit t d W / 4 (shifted by 16
  // for odd t when the run is not a whole number of words); q8_0: bytes 8t .. 8t + 7 of each block.
  static constexpr int KBits = KQ8 ? 0 : D * WK / 4;
  static constexpr int KLoad = KQ8 ? D / 16 : cover_words(KBits, 4);
  static constexpr int KRun = KQ8 ? 1 : (KBits + 31) / 32;
  static constexpr bool KShift = !KQ8 && KBits % 32 != 0;
  static constexpr int KVec = KQ8 ? 8 : (KShift ? 4 : vec_bytes(KPay, KBits / 8));
  static constexpr int KHdrW = KQ8 ? D / 64 : 1;  // 32-bit header words per token
  // V words per thread and token.  turbo: the d W / 8-bit run at bit g d W / 8; q8_0: bytes
  // g d/8 .. (g+1) d/8 - 1.
  static constexpr int VBits = VQ8 ? 0 : D * WV / 8;
  static constexpr int VLoad = VQ8 ? D / 32 : cover_words(VBits, 8);
  static constexpr int VRun = VQ8 ? 1 : (VBits + 31) / 32;
  static constexpr bool VShift = !VQ8 && VBits % 32 != 0;
  static constexpr int VVec = VQ8 ? vec_bytes(VPay, D / 8) : (VShift ? 4 : vec_bytes(VPay, VBits / 8));
  // Tables: K entries 8 B x 32 lanes, V entries 4 B x 32 lanes, each aligned to its own size.
  static constexpr uint32_t KLut = KQ8 ? 0u : (256u << (2 * WK));
  static constexpr uint32_t VLut = VQ8 ? 0u : (128u << (2 * WV));
  static constexpr uint32_t Big = KLut > VLut ? KLut : VLut, Small = KLut > VLut ? VLut : KLut;
};

// Launch shape of one kernel: NQ 8-column products per part (1: up to 4 query heads per KV head as
// high / low parts, 2: up to 8, 4: up to 16); per warp a block of P' tiles and the query fragments (8 bytes per lane, product
// and k step); the two tables.  Shared layout (attend_mma_kernel): the larger table on the first
// boundary of its size, the smaller table right below it (else right above), as many warp blocks
// as fit below that from the start, the others above the tables; whatever the start's alignment,
// that ends within Big + Small + warps * block + max(Small, block) bytes, or 2 Big + Small when the
// gap below the larger table holds every warp block.  16 warps (d = 256: 8, for its ~180
// registers a thread), halved until the shared memory fits.
constexpr int kSmemLimit = 227 * 1024;
template <class F, int NQ_>
struct Shape {
  static constexpr int NQ = NQ_;
  static constexpr bool HILO = NQ == 1;
  static constexpr int NV = HILO ? 1 : NQ / 2;  // 8-column V products (P' tiles) per tile
  // Tiles a warp works on at once: two (two independent chains of loads, lookups and products,
  // one query-fragment read for both) where the registers allow it, that is with up to 4 query
  // heads per KV head at d <= 128, run with 12 warps of up to 168 registers; else one.
  static constexpr int NT = (HILO && F::D <= 128) ? 2 : 1;
  static constexpr int QfBytes = F::KS * 256 * (F::KQ8 ? 1 : 2) * NQ;
  static constexpr int PsBytes = 512 * NT * NV;
  static constexpr int Block = PsBytes + QfBytes;
  // turbo-MSE V of 2 or 3 bits with up to 4 query heads: a 64 KB V table of byte-indexed entries
  // (two tables in one: the code pair in a byte's low bits at + 0, in its high bits at + 128), so
  // that every lookup address is one byte permute of the codes (accumulate_v)
  static constexpr bool DualV = HILO && !F::VQ8 && (F::WV == 2 || F::WV == 3);
  static constexpr uint32_t VLut = DualV ? 65536u : F::VLut;
  static constexpr uint32_t Big = F::KLut > VLut ? F::KLut : VLut, Small = F::KLut > VLut ? VLut : F::KLut;
  static constexpr int smem(int warps) {
    if (Small == Big) {  // the second table right above the first; warp blocks below, then above
      const int blocks = (warps + 1) * Block;
      return (int)(2 * Big) + (blocks > (int)Big ? blocks : (int)Big);
    }
    const int packed = (int)(Big + Small) + warps * Block + ((int)Small > Block ? (int)Small : Block);
    const int gap = (int)(2 * Big + Small);
    return packed > gap ? packed : gap;
  }
  static constexpr int W0 = F::D == 256 ? 8 : (NT == 2 ? 12 : (NQ == 4 ? 8 : 16));
  static constexpr int Warps = smem(W0) <= kSmemLimit ? W0 : smem(W0 / 2) <= kSmemLimit ? W0 / 2 : W0 / 4;
  static constexpr int Threads = 32 * Warps;
  static constexpr int Smem = smem(Warps);
  static_assert(Smem <= kSmemLimit, "shared memory");
};

// Loads N consecutive words from p (VEC-byte aligned) with the evict-first policy.
template <int N, int VEC>
__device__ __forceinline__ void load_words(uint32_t (&w)[N], const unsigned char* p, uint64_t pol) {
  if constexpr (VEC == 16 && N % 4 == 0) {
#pragma unroll
    for (int j = 0; j < N; j += 4) {
      const uint4 v = ld_stream_v4(p + 4 * j, pol);
      w[j] = v.x; w[j + 1] = v.y; w[j + 2] = v.z; w[j + 3] = v.w;
    }
  } else if constexpr (VEC >= 8 && N % 2 == 0) {
#pragma unroll
    for (int j = 0; j < N; j += 2) {
      const uint2 v = ld_stream_v2(p + 4 * j, pol);
      w[j] = v.x; w[j + 1] = v.y;
    }
  } else {
#pragma unroll
    for (int j = 0; j < N; ++j) w[j] = ld_stream_u32(p + 4 * j, pol);
  }
}

// The run of bits that starts at bit sh of w[0] (sh < 32), as words from bit 0.
template <int NL, int NR, bool SHIFT>
__device__ __forceinline__ void make_run(const uint32_t (&w)[NL], uint32_t (&r)[NR], uint32_t sh) {
#pragma unroll
  for (int j = 0; j < NR; ++j) {
    if constexpr (SHIFT) r[j] = j + 1 < NL ? __funnelshift_r(w[j], w[j + 1 < NL ? j + 1 : j], sh) : (w[j] >> sh);
    else r[j] = w[j];
  }
}

// Table address for the N bits at bit p of the run r: base | bits << SH (p a constant once the
// caller's loop is unrolled; base has zeros in bits SH .. SH + N - 1).  A whole byte at bit 8 of
// a base whose bits 8 .. 15 are zero is one byte permute.
template <int N, int SH, int NR>
__device__ __forceinline__ uint32_t run_addr(const uint32_t (&r)[NR], int p, uint32_t base) {
  const int wi = p >> 5, off = p & 31;
  if (N == 8 && SH == 8 && (off & 7) == 0) return __byte_perm(r[wi], base, 0x7604u | ((uint32_t)(off >> 3) << 4));
  uint32_t x;
  if (off + N <= 32) x = off >= SH ? (r[wi] >> (off - SH)) : (r[wi] << (SH - off));
  else if (off >= SH) x = __funnelshift_r(r[wi], r[wi + 1 < NR ? wi + 1 : wi], off - SH);
  else x = __funnelshift_r(r[wi], r[wi + 1 < NR ? wi + 1 : wi], off) << SH;
  return (x & (((1u << N) - 1u) << SH)) | base;
}

struct Cursor {
  const unsigned char *kp, *kh, *vp, *vh;  // this lane's addresses in the current tile
  int in_page, page_ord;                   // token offset in its page; logical page
  bool ok;                                 // page in range
};

template <class F, int NQ>
struct MmaWarp {
  static constexpr int D = F::D, KS = F::KS;
  static constexpr bool HILO = NQ == 1;
  // head slots per thread (heads t, t + 4, t + 8, t + 12) = 8-column products per part; V products
  static constexpr int NH = NQ, NV = Shape<F, NQ>::NV;
  static constexpr bool DualV = Shape<F, NQ>::DualV;

  struct KTile {
    uint32_t a[F::KLoad], b[F::KLoad];  // tokens g, g + 8
    uint32_t ha[F::KHdrW], hb[F::KHdrW];
  };
  struct VTile {
    uint32_t w[4][F::VLoad];  // tokens t, t + 8, t + 4, t + 12
    uint32_t h0, h1;          // turbo: norms of tokens g, g + 8; q8_0: scales of t, t + 8 and t + 4, t + 12
  };

  const DecodeLaunch& k;
  int lane, g, t;
  uint32_t ylk, ylv;         // table bases | lane offsets
  uint32_t psw0, psw1, psr;  // shared addresses of this lane's P' words in the warp's first P' tile
  uint32_t qf;               // shared address of this lane's query fragments
  uint32_t ksh, vsh;         // bit offsets of the K and V runs in their first words
  int kto, vgo;              // byte offsets of this lane's K and V words in a vector
  int vhdr;                  // byte offset of this lane's V header entry (q8_0: its block's scale)
  int vwo[F::VLoad];         // byte offsets of the V words from the first (clamped to the payload)
  bool pf_k, pf_v, pf_h;     // bulk prefetch allowed (16-byte aligned tile starts)
  uint64_t pol;              // cache loads: evict first
  uint64_t pol_keep;         // partials: evict last (the combine reads them from L2, then drops them)

  int layer, layer_v, b, kvh, ntiles, last_valid;  // layer: of the K view; layer_v: of the V view
  int gof, gcn;  // this item's query heads: [gof, gof + gcn) of the KV head's G
  Cursor c;
  KTile kn[2];  // the next pair's K and V, loaded one phase ahead (pipelined pair steps)
  VTile vn[2];
  // V accumulators of product v: entries 0, 1 = row g, columns 2t, 2t + 1; 2, 3 = row g + 8.  Up to
  // 4 heads: the columns are head t's high and low parts; more: column 2t = head slot 2v (head
  // t + 8v), column 2t + 1 = head slot 2v + 1 (head t + 8v + 4).
  float oacc[NV][KS][4];
  float m[NH], l[NH];

  __device__ __forceinline__ MmaWarp(const DecodeLaunch& k_) : k(k_) {}

  __device__ __forceinline__ void init_lane(int lane_) {
    lane = lane_;
    g = lane >> 2;
    t = lane & 3;
    if constexpr (F::KQ8) {
      kto = 8 * t;
      ksh = 0;
    } else {
      kto = 4 * ((t * F::KBits) >> 5);
      ksh = (uint32_t)(t * F::KBits) & 31u;
    }
    if constexpr (F::VQ8) {
      vgo = g * (D / 8);
      vsh = 0;
      vhdr = 2 * ((g * (D / 8)) >> 5);
#pragma unroll
      for (int j = 0; j < F::VLoad; ++j) vwo[j] = 4 * j;
    } else {
      const int w0 = (g * F::VBits) >> 5, last = F::VPay / 4 - 1;
      vgo = 4 * w0;
      vsh = (uint32_t)(g * F::VBits) & 31u;
      vhdr = 0;
#pragma unroll
      for (int j = 0; j < F::VLoad; ++j) vwo[j] = 4 * (min(w0 + j, last) - w0);
    }
    const DecodeArgs& a = k.a;
    const bool pg16 = a.k.page_size % 16 == 0;
    pf_k = pg16 || F::KPay % 16 == 0;
    pf_v = pg16 || F::VPay % 16 == 0;
    pf_h = pg16 && ((reinterpret_cast<uintptr_t>(a.k.header) | reinterpret_cast<uintptr_t>(a.v.header)) & 15) == 0;
  }

  __device__ __forceinline__ void set_page(Cursor& cu) {
    const DecodeArgs& a = k.a;
    long long page = b;
    cu.ok = true;
    if (a.block_table) {
      page = a.block_table[(long long)b * a.max_blocks_per_seq + cu.page_ord];
      if (page < 0 || page >= a.k.num_pages) {
        if (lane == 0) atomicOr(k.tab.status, kFlagBlockTable);
        cu.ok = false;
        page = 0;
      }
    }
    const long long pv = ((long long)page * a.k.H + kvh) * a.k.page_size + cu.in_page;  // vector in its layer
    const long long lv = (long long)a.k.num_pages * a.k.H * a.k.page_size;               // vectors per layer
    const long long base = layer * lv + pv, vbase = layer_v * lv + pv;
    cu.kp = a.k.payload + (base + g) * F::KPay + kto;
    cu.kh = a.k.header + (base + g) * F::KHdr;
    cu.vp = a.v.payload + (vbase + t) * F::VPay + vgo;
    cu.vh = F::VQ8 ? a.v.header + (vbase + t) * F::VHdr + vhdr : a.v.header + (vbase + g) * F::VHdr;
  }

  __device__ __forceinline__ void advance(Cursor& cu) {
    cu.in_page += 16;
    if (cu.in_page == k.a.k.page_size) {
      cu.in_page = 0;
      ++cu.page_ord;
      set_page(cu);
    } else {
      cu.kp += 16 * F::KPay;
      cu.kh += 16 * F::KHdr;
      cu.vp += 16 * F::VPay;
      cu.vh += 16 * F::VHdr;
    }
  }

  // Rows at or beyond nvalid (ragged last tile) re-read row nvalid - 1; their scores are masked.
  // FULL: a whole tile, every row offset a constant.
  template <bool FULL>
  __device__ __forceinline__ void load_k(KTile& K, const Cursor& c, int nvalid) {
    int da = 0, db = 8;
    if (!FULL) {
      da = min(g, nvalid - 1) - g;
      db = min(g + 8, nvalid - 1) - g;
    }
    const unsigned char* pa = c.kp + da * F::KPay;
    const unsigned char* pb = c.kp + db * F::KPay;
    if constexpr (F::KQ8) {
#pragma unroll
      for (int blk = 0; blk < D / 32; ++blk) {
        const uint2 x = ld_stream_v2(pa + 32 * blk, pol), y = ld_stream_v2(pb + 32 * blk, pol);
        K.a[2 * blk] = x.x; K.a[2 * blk + 1] = x.y;
        K.b[2 * blk] = y.x; K.b[2 * blk + 1] = y.y;
      }
    } else {
      load_words<F::KLoad, F::KVec>(K.a, pa, pol);
      load_words<F::KLoad, F::KVec>(K.b, pb, pol);
    }
#pragma unroll
    for (int j = 0; j < F::KHdrW; ++j) {
      K.ha[j] = ld_stream_u32(c.kh + da * F::KHdr + 4 * j, pol);
      K.hb[j] = ld_stream_u32(c.kh + db * F::KHdr + 4 * j, pol);
    }
  }

  template <bool FULL>
  __device__ __forceinline__ void load_v(VTile& V, const Cursor& c, int nvalid) {
    const int rows[4] = {t, t + 8, t + 4, t + 12};
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const int dr = !FULL ? min(rows[r], nvalid - 1) - t : rows[r] - t;
      const unsigned char* p = c.vp + dr * F::VPay;
      if constexpr (F::VQ8 || F::VLoad == 1 || !F::VShift) {
        load_words<F::VLoad, F::VVec>(V.w[r], p, pol);
      } else {
#pragma unroll
        for (int j = 0; j < F::VLoad; ++j) V.w[r][j] = ld_stream_u32(p + vwo[j], pol);
      }
    }
    if constexpr (F::VQ8) {
      uint32_t s[4];
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const int dr = !FULL ? min(rows[r], nvalid - 1) - t : rows[r] - t;
        s[r] = ld_stream_u16(c.vh + dr * F::VHdr, pol);
      }
      V.h0 = s[0] | (s[1] << 16);
      V.h1 = s[2] | (s[3] << 16);
#pragma unroll
      for (int r = 0; r < 4; ++r) {
#pragma unroll
        for (int j = 0; j < F::VLoad; ++j) V.w[r][j] ^= 0x80808080u;
      }
    } else {
      const int da = !FULL ? min(g, nvalid - 1) - g : 0;
      const int db = !FULL ? min(g + 8, nvalid - 1) - g : 8;
      V.h0 = ld_stream_u16(c.vh + da * F::VHdr, pol) | (ld_stream_u16(c.vh + db * F::VHdr, pol) << 16);
      V.h1 = 0;
    }
  }

  // Requests tiles [tile + ahead, tile + ahead + n) into L2, n <= count, clipped to the work
  // item and to the page (lane 0, whose addresses are the current tile's own).
  __device__ __forceinline__ void prefetch_tiles(int tile, int ahead, int count) {
    const int n = min(min(ntiles - tile - ahead, count), (k.a.k.page_size - c.in_page) / 16 - ahead);
    if (lane != 0 || n <= 0 || !c.ok) return;
    if (pf_k) prefetch_l2(c.kp + 16 * ahead * F::KPay, 16 * n * F::KPay);
    if (pf_v) prefetch_l2(c.vp + 16 * ahead * F::VPay, 16 * n * F::VPay);
    if (pf_h) {
      prefetch_l2(c.kh + 16 * ahead * F::KHdr, 16 * n * F::KHdr);
      prefetch_l2(c.vh + 16 * ahead * F::VHdr, 16 * n * F::VHdr);
    }
  }

  // Raises the reference of every head whose new scores pass it by 2^8 (warp-uniform decision).
  __device__ __forceinline__ void raise_reference(float (&mx)[NH]) {
    bool need = false;
#pragma unroll
    for (int h = 0; h < NH; ++h) need |= mx[h] > m[h] + kLazyMax;
    if (!__any_sync(kFull, need)) return;
#pragma unroll
    for (int h = 0; h < NH; ++h) {
#pragma unroll
      for (int o = 4; o < 32; o <<= 1) mx[h] = fmaxf(mx[h], __shfl_xor_sync(kFull, mx[h], o));
      const float mn = fmaxf(m[h], mx[h]);
      const float al = ex2(m[h] - mn);
      l[h] *= al;
#pragma unroll
      for (int mt = 0; mt < KS; ++mt) {
        if (HILO) {
#pragma unroll
          for (int e = 0; e < 4; ++e) oacc[0][mt][e] *= al;
        } else {
          oacc[h >> 1][mt][h & 1] *= al;
          oacc[h >> 1][mt][2 + (h & 1)] *= al;
        }
      }
      m[h] = mn;
    }
  }

  // Score products of NT tiles: cc[j][q] = codebook (or int8) part, cs[j][q] = QJL part of tile j
  // and heads 4q .. 4q + 3 (columns 2h / 2h + 1 = high / low part of head 4q + h).  Query
  // fragments of head block q and step ch (read once for all NT tiles): turbo K at
  // qf + 512 (KS q + ch), 16 bytes a lane (the q' pair, then the S q' pair); q8_0 at
  // qf + 256 (KS q + ch), 8 bytes a lane.  A turbo K table entry holds the codebook pair of each
  // lane at lane * 4 and the sign pair at 128 + lane * 4, so both reads of a lookup share one
  // address and land in the product's operand registers directly.
  template <int NT>
  __device__ __forceinline__ void score(const KTile (&K)[NT], float (&cc)[NT][NH][4], float (&cs)[NT][NH][4]) {
    if constexpr (F::KQ8) {
#pragma unroll
      for (int blk = 0; blk < D / 32; ++blk) {
        uint2 f0[NH], f1[NH];
#pragma unroll
        for (int q = 0; q < NH; ++q) {
          f0[q] = lds64(qf + 256 * (KS * q + 2 * blk));
          f1[q] = lds64(qf + 256 * (KS * q + 2 * blk + 1));
        }
#pragma unroll
        for (int j = 0; j < NT; ++j) {
          const uint32_t xa0 = K[j].a[2 * blk] ^ 0x80808080u, xa1 = K[j].a[2 * blk + 1] ^ 0x80808080u;
          const uint32_t xb0 = K[j].b[2 * blk] ^ 0x80808080u, xb1 = K[j].b[2 * blk + 1] ^ 0x80808080u;
          const uint32_t a00 = i8x2_to_h2<0x4140>(xa0), a01 = i8x2_to_h2<0x4140>(xb0);
          const uint32_t a02 = i8x2_to_h2<0x4342>(xa0), a03 = i8x2_to_h2<0x4342>(xb0);
          const uint32_t a10 = i8x2_to_h2<0x4140>(xa1), a11 = i8x2_to_h2<0x4140>(xb1);
          const uint32_t a12 = i8x2_to_h2<0x4342>(xa1), a13 = i8x2_to_h2<0x4342>(xb1);
          const int sh = 16 * (blk & 1);
          const float da = __half2float(__ushort_as_half((unsigned short)(K[j].ha[blk >> 1] >> sh)));
          const float db = __half2float(__ushort_as_half((unsigned short)(K[j].hb[blk >> 1] >> sh)));
#pragma unroll
          for (int q = 0; q < NH; ++q) {
            float c[4];
            mma_16816_zc(c, a00, a01, a02, a03, f0[q].x, f0[q].y);
            mma_16816(c, a10, a11, a12, a13, f1[q].x, f1[q].y);
            cc[j][q][0] = fmaf(da, c[0], cc[j][q][0]);
            cc[j][q][1] = fmaf(da, c[1], cc[j][q][1]);
            cc[j][q][2] = fmaf(db, c[2], cc[j][q][2]);
            cc[j][q][3] = fmaf(db, c[3], cc[j][q][3]);
          }
        }
      }
    } else {
      constexpr int N = 2 * F::WK;
      uint32_t ra[NT][F::KRun], rb[NT][F::KRun];
#pragma unroll
      for (int j = 0; j < NT; ++j) {
        make_run<F::KLoad, F::KRun, F::KShift>(K[j].a, ra[j], ksh);
        make_run<F::KLoad, F::KRun, F::KShift>(K[j].b, rb[j], ksh);
      }
#pragma unroll
      for (int ch = 0; ch < KS; ++ch) {
        const int p = 4 * ch * F::WK;
        uint4 f[NH];
#pragma unroll
        for (int q = 0; q < NH; ++q) f[q] = lds128(qf + 512 * (KS * q + ch));  // q' high/low, then S q'
#pragma unroll
        for (int j = 0; j < NT; ++j) {
          const uint32_t aa0 = run_addr<N, 8>(ra[j], p, ylk), aa1 = run_addr<N, 8>(ra[j], p + N, ylk);
          const uint32_t ab0 = run_addr<N, 8>(rb[j], p, ylk), ab1 = run_addr<N, 8>(rb[j], p + N, ylk);
#pragma unroll
          for (int q = 0; q < NH; ++q) {
            mma_16816(cc[j][q], lds32(aa0), lds32(ab0), lds32(aa1), lds32(ab1), f[q].x, f[q].y);
            mma_16816(cs[j][q], lds32(aa0 + 128), lds32(ab0 + 128), lds32(aa1 + 128), lds32(ab1 + 128), f[q].z,
                      f[q].w);
          }
        }
      }
    }
  }

  // V products of a tile with the P' fragments bp[v] of product v.
  __device__ __forceinline__ void accumulate_v(const VTile& V, const uint2 (&bp)[NV]) {
    if constexpr (F::VQ8) {
      const __half2 d01 = u32_as_h2(V.h0), d23 = u32_as_h2(V.h1);
#pragma unroll
      for (int mt = 0; mt < KS; ++mt) {
        const int wi = (2 * mt) >> 2;
        const uint32_t sel = (mt & 1) ? 0x7362u : 0x5140u;  // bytes 2mt, 2mt + 1 of two tokens
        const uint32_t x01 = __byte_perm(V.w[0][wi], V.w[1][wi], sel);
        const uint32_t x23 = __byte_perm(V.w[2][wi], V.w[3][wi], sel);
        const uint32_t a0 = h2_as_u32(__hmul2(u32_as_h2(i8x2_to_h2<0x4140>(x01)), d01));
        const uint32_t a1 = h2_as_u32(__hmul2(u32_as_h2(i8x2_to_h2<0x4342>(x01)), d01));
        const uint32_t a2 = h2_as_u32(__hmul2(u32_as_h2(i8x2_to_h2<0x4140>(x23)), d23));
        const uint32_t a3 = h2_as_u32(__hmul2(u32_as_h2(i8x2_to_h2<0x4342>(x23)), d23));
#pragma unroll
        for (int v = 0; v < NV; ++v) mma_16816(oacc[v][mt], a0, a1, a2, a3, bp[v].x, bp[v].y);
      }
    } else {
      constexpr int N = 2 * F::WV;
      uint32_t r[4][F::VRun];
#pragma unroll
      for (int q = 0; q < 4; ++q) make_run<F::VLoad, F::VRun, F::VShift>(V.w[q], r[q], vsh);
      // byte-indexed table (3 bits: the run and the run shifted by 4 bits give every pair of
      // coordinates as the low or high 6 bits of a byte; 2 bits: as a byte's low or high nibble)
      uint32_t r4[4][F::VRun];
      if constexpr (DualV && F::WV == 3) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
#pragma unroll
          for (int j = 0; j < F::VRun; ++j)
            r4[q][j] = j + 1 < F::VRun ? __funnelshift_r(r[q][j], r[q][j + 1 < F::VRun ? j + 1 : j], 4) : r[q][j] >> 4;
        }
      }
#pragma unroll
      for (int mt = 0; mt < KS; ++mt) {
        uint32_t e[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          if constexpr (DualV) {
            // pair mt: byte, half (high: + 128) and source (the run or the run >> 4)
            int byte, hi;
            bool shifted = false;
            if constexpr (F::WV == 3) {
              const int m = mt >> 2, i = mt & 3;
              byte = 3 * m + (i == 2 ? 1 : i == 3 ? 2 : 0);
              hi = i & 1;
              shifted = i == 1 || i == 2;
            } else {
              byte = mt >> 1;
              hi = mt & 1;
            }
            const uint32_t src = shifted ? r4[q][byte >> 2] : r[q][byte >> 2];
            e[q] = lds32(__byte_perm(src, ylv, 0x7604u | ((uint32_t)(byte & 3) << 4)) + 128u * hi);
          } else {
            e[q] = lds32(run_addr<N, 7>(r[q], 2 * mt * F::WV, ylv));
          }
        }
        // a0/a1: slots 2t, 2t+1 = tokens t, t+8 at coordinate 2mt / 2mt+1; a2/a3: tokens t+4, t+12
        const uint32_t a0 = __byte_perm(e[0], e[1], 0x5410), a1 = __byte_perm(e[0], e[1], 0x7632);
        const uint32_t a2 = __byte_perm(e[2], e[3], 0x5410), a3 = __byte_perm(e[2], e[3], 0x7632);
#pragma unroll
        for (int v = 0; v < NV; ++v) mma_16816(oacc[v][mt], a0, a1, a2, a3, bp[v].x, bp[v].y);
      }
    }
  }

  // NT tiles at the cursors cu[0 .. NT - 1] (consecutive tiles of the work item, pages in range);
  // the last one holds nlast valid rows (a whole tile when FULLLAST).  P' tiles at kBuf + 256 j
  // in the warp's P' block.  Whole tiles run with constant row offsets.
  template <int NT, bool FULLLAST>
  __device__ __forceinline__ void step_tiles(const Cursor (&cu)[NT], int nlast, uint32_t kBuf) {
    KTile kc[NT];
    VTile vc[NT];
#pragma unroll
    for (int j = 0; j < NT; ++j) {
      if (j < NT - 1 || FULLLAST) load_k<true>(kc[j], cu[j], 16);
      else load_k<false>(kc[j], cu[j], nlast);
    }
    // Up to 4 query heads: V loads in flight with K's (one load latency per tile); with two
    // products per part the registers are short, and V is loaded after the score products.
    if constexpr (HILO) {
#pragma unroll
      for (int j = 0; j < NT; ++j) {
        if (j < NT - 1 || FULLLAST) load_v<true>(vc[j], cu[j], 16);
        else load_v<false>(vc[j], cu[j], nlast);
      }
    }
    float cc[NT][NH][4], cs[NT][NH][4];
#pragma unroll
    for (int j = 0; j < NT; ++j) {
#pragma unroll
      for (int q = 0; q < NH; ++q) {
#pragma unroll
        for (int e = 0; e < 4; ++e) cc[j][q][e] = cs[j][q][e] = 0.f;
      }
    }
    score<NT>(kc, cc, cs);
    if constexpr (!HILO) {
#pragma unroll
      for (int j = 0; j < NT; ++j) {
        if (j < NT - 1 || FULLLAST) load_v<true>(vc[j], cu[j], 16);
        else load_v<false>(vc[j], cu[j], nlast);
      }
    }

    // thread (g, t) and head slot h (head t + 4h): entries 0, 1 of product h = token g, the
    // high and low parts; entries 2, 3 = token g + 8.
    float s[NT][NH][2];
#pragma unroll
    for (int j = 0; j < NT; ++j) {
      if constexpr (F::KQ8) {
#pragma unroll
        for (int h = 0; h < NH; ++h) {
          s[j][h][0] = cc[j][h][0] + cc[j][h][1];
          s[j][h][1] = cc[j][h][2] + cc[j][h][3];
        }
      } else {
        const float2 hA = __half22float2(u32_as_h2(kc[j].ha[0])), hB = __half22float2(u32_as_h2(kc[j].hb[0]));
#pragma unroll
        for (int h = 0; h < NH; ++h) {
          s[j][h][0] = fmaf(hA.x, cc[j][h][0] + cc[j][h][1], hA.y * (cs[j][h][0] + cs[j][h][1]));
          s[j][h][1] = fmaf(hB.x, cc[j][h][2] + cc[j][h][3], hB.y * (cs[j][h][2] + cs[j][h][3]));
        }
      }
    }
    if (!FULLLAST) {
#pragma unroll
      for (int h = 0; h < NH; ++h) {
        if (g >= nlast) s[NT - 1][h][0] = -INFINITY;
        if (g + 8 >= nlast) s[NT - 1][h][1] = -INFINITY;
      }
    }

    // ---- online softmax with a lazily raised reference (base 2) ----
    {
      float mx[NH];
#pragma unroll
      for (int h = 0; h < NH; ++h) {
        mx[h] = fmaxf(s[0][h][0], s[0][h][1]);
#pragma unroll
        for (int j = 1; j < NT; ++j) mx[h] = fmaxf(mx[h], fmaxf(s[j][h][0], s[j][h][1]));
      }
      raise_reference(mx);
    }
    float p[NT][NH][2];
#pragma unroll
    for (int j = 0; j < NT; ++j) {
#pragma unroll
      for (int h = 0; h < NH; ++h) {
        p[j][h][0] = ex2(s[j][h][0] - m[h]);
        p[j][h][1] = ex2(s[j][h][1] - m[h]);
        l[h] += p[j][h][0] + p[j][h][1];
      }
    }
    // ---- Sparse V: weights below the threshold are dropped; a step whose weights are all
    // dropped skips V ----
    if (k.a.skip_threshold > 0.f) {
      const float tau = k.a.skip_threshold;
      bool any = false;
#pragma unroll
      for (int j = 0; j < NT; ++j) {
#pragma unroll
        for (int h = 0; h < NH; ++h) {
          p[j][h][0] = p[j][h][0] >= tau ? p[j][h][0] : 0.f;
          p[j][h][1] = p[j][h][1] >= tau ? p[j][h][1] : 0.f;
          any |= (p[j][h][0] + p[j][h][1]) > 0.f;
        }
      }
      if (!__any_sync(kFull, any)) {
        __syncwarp();
        return;
      }
    }

    // ---- P' = weight (* V norm for turbo V), one word per (column, token pair g / g + 8) ----
#pragma unroll
    for (int j = 0; j < NT; ++j) {
      float2 nv = make_float2(1.f, 1.f);
      if constexpr (!F::VQ8) nv = __half22float2(u32_as_h2(vc[j].h0));
      if (HILO) {
        const uint32_t buf = kBuf + 256 * j;
        const float w0 = p[j][0][0] * nv.x, w1 = p[j][0][1] * nv.y;
        const __half2 hi = __floats2half2_rn(w0, w1);
        const float2 hf = __half22float2(hi);
        sts32(psw0 + buf, h2_as_u32(hi));
        sts32(psw1 + buf, h2_as_u32(__floats2half2_rn(w0 - hf.x, w1 - hf.y)));
      } else {
#pragma unroll
        for (int v = 0; v < NV; ++v) {  // P' tile v: head slots 2v (column 2t) and 2v + 1 (column 2t + 1)
          const uint32_t buf = kBuf + 256 * (j * NV + v);
          sts32(psw0 + buf, h2_as_u32(__floats2half2_rn(p[j][2 * v][0] * nv.x, p[j][2 * v][1] * nv.y)));
          sts32(psw1 + buf,
                h2_as_u32(__floats2half2_rn(p[j][2 * v + 1][0] * nv.x, p[j][2 * v + 1][1] * nv.y)));
        }
      }
    }
    __syncwarp();
#pragma unroll
    for (int j = 0; j < NT; ++j) {
      uint2 bp[NV];
#pragma unroll
      for (int v = 0; v < NV; ++v) bp[v] = lds64_v(psr + kBuf + 256 * (j * NV + v));
      accumulate_v(vc[j], bp);
    }
  }

  // A pair of whole tiles whose K and V were loaded into kn / vn by the previous step; their
  // cursors cu (a tile whose page is out of range has its scores masked: its loads read page 0).
  // With MORE, the next pair's loads (cursors nx) are issued into kn as soon as the score
  // products have consumed K, and into vn once the V products have consumed V, so each load has
  // about half a step to land before it is needed.
  template <bool MORE>
  __device__ __forceinline__ void step_pipelined(const Cursor (&cu)[2], const Cursor (&nx)[2], uint32_t kBuf) {
    KTile kc[2] = {kn[0], kn[1]};
    VTile vc[2] = {vn[0], vn[1]};
    float cc[2][NH][4], cs[2][NH][4];
#pragma unroll
    for (int j = 0; j < 2; ++j) {
#pragma unroll
      for (int q = 0; q < NH; ++q) {
#pragma unroll
        for (int e = 0; e < 4; ++e) cc[j][q][e] = cs[j][q][e] = 0.f;
      }
    }
    score<2>(kc, cc, cs);
    if (MORE) {
      load_k<true>(kn[0], nx[0], 16);
      load_k<true>(kn[1], nx[1], 16);
    }
    float s[2][NH][2];
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const float2 hA = __half22float2(u32_as_h2(kc[j].ha[0])), hB = __half22float2(u32_as_h2(kc[j].hb[0]));
#pragma unroll
      for (int h = 0; h < NH; ++h) {
        if constexpr (F::KQ8) {
          s[j][h][0] = cc[j][h][0] + cc[j][h][1];
          s[j][h][1] = cc[j][h][2] + cc[j][h][3];
        } else {
          s[j][h][0] = fmaf(hA.x, cc[j][h][0] + cc[j][h][1], hA.y * (cs[j][h][0] + cs[j][h][1]));
          s[j][h][1] = fmaf(hB.x, cc[j][h][2] + cc[j][h][3], hB.y * (cs[j][h][2] + cs[j][h][3]));
        }
        if (!cu[j].ok) s[j][h][0] = s[j][h][1] = -INFINITY;  // warp-uniform
      }
    }
    float mx[NH];
#pragma unroll
    for (int h = 0; h < NH; ++h) mx[h] = fmaxf(fmaxf(s[0][h][0], s[0][h][1]), fmaxf(s[1][h][0], s[1][h][1]));
    raise_reference(mx);
    float p[2][NH][2];
    bool any = false;
#pragma unroll
    for (int j = 0; j < 2; ++j) {
#pragma unroll
      for (int h = 0; h < NH; ++h) {
        p[j][h][0] = ex2(s[j][h][0] - m[h]);
        p[j][h][1] = ex2(s[j][h][1] - m[h]);
        l[h] += p[j][h][0] + p[j][h][1];
      }
    }
    // Sparse V: weights below the threshold are dropped; a pair whose weights are all dropped
    // skips the V products (its next V loads are issued all the same)
    const float tau = k.a.skip_threshold;
    if (tau > 0.f) {
#pragma unroll
      for (int j = 0; j < 2; ++j) {
#pragma unroll
        for (int h = 0; h < NH; ++h) {
          p[j][h][0] = p[j][h][0] >= tau ? p[j][h][0] : 0.f;
          p[j][h][1] = p[j][h][1] >= tau ? p[j][h][1] : 0.f;
          any |= (p[j][h][0] + p[j][h][1]) > 0.f;
        }
      }
    }
    if (tau <= 0.f || __any_sync(kFull, any)) {
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        float2 nv = make_float2(1.f, 1.f);
        if constexpr (!F::VQ8) nv = __half22float2(u32_as_h2(vc[j].h0));
        const uint32_t buf = kBuf + 256 * j;
        const float w0 = p[j][0][0] * nv.x, w1 = p[j][0][1] * nv.y;
        const __half2 hi = __floats2half2_rn(w0, w1);
        const float2 hf = __half22float2(hi);
        sts32(psw0 + buf, h2_as_u32(hi));
        sts32(psw1 + buf, h2_as_u32(__floats2half2_rn(w0 - hf.x, w1 - hf.y)));
      }
      __syncwarp();
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const uint2 bp[1] = {lds64_v(psr + kBuf + 256 * j)};
        accumulate_v(vc[j], bp);
      }
    }
    __syncwarp();
    if (MORE) {
      load_v<true>(vn[0], nx[0], 16);
      load_v<true>(vn[1], nx[1], 16);
    }
  }

  // One tile at cursor cu, skipped when its page is out of range.
  __device__ __forceinline__ void step_one(const Cursor& cu, bool last, uint32_t kBuf) {
    if (!cu.ok) {  // warp-uniform
      __syncwarp();
      return;
    }
    const Cursor one[1] = {cu};
    if (last && last_valid < 16) step_tiles<1, false>(one, last_valid, kBuf);
    else step_tiles<1, true>(one, 16, kBuf);
  }

  __device__ __forceinline__ void run_item(unsigned int item) {
    const DecodeArgs& a = k.a;
    const int H = a.k.H, G = k.G, Hq = a.n_q_heads;
    gof = k.g_off;
    gcn = k.g_cnt;
    if (k.g_halves == 2) {  // consecutive counter values: the two head halves of one item
      const bool hi = item & 1u;
      item >>= 1;
      gof = hi ? k.g_cnt : 0;
      gcn = hi ? G - k.g_cnt : k.g_cnt;
    }
    const int split = (int)(item % k.n_splits);
    const unsigned int rest = item / k.n_splits;
    kvh = (int)(rest % H);
    const int lb = (int)(rest / H);
    layer = k_layer_of(a, lb / a.batch);
    layer_v = v_layer_of(a, lb / a.batch);
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

    // ---- B fragments of product q, column g: head 4q + g/2, the high (g even) or low (g odd)
    // fp16 part.  k slots 2t, 2t + 1 (+8) of step ch = the coordinates c0(ch) + {0, 1} ({2, 3})
    // that the A fragments hold.  Codebook (or int8) product: q' with log2 e (/ lambda for turbo
    // K); QJL product: S q' with log2 e sqrt(pi/2) / d ----
#pragma unroll
    for (int q = 0; q < NH; ++q) {
      const int head = 4 * q + (g >> 1);
      const bool lo = g & 1;
      const bool valid = head < gcn;
      const float* qp = k.qprep + (row0 + gof + (valid ? head : 0)) * 2 * D;
      const float fq = valid ? (F::KQ8 ? kLog2e : kLog2e / k.tab.f16_scale[F::KQ8 ? 0 : F::WK - 2]) : 0.f;
      const float fs = valid ? kLog2e * kSqrtHalfPi / (float)D : 0.f;
#pragma unroll
      for (int ch = 0; ch < KS; ++ch) {
        const int c0 = F::KQ8 ? 32 * (ch >> 1) + 8 * t + 4 * (ch & 1) : t * (D / 4) + 4 * ch;
        const float4 v = *reinterpret_cast<const float4*>(qp + c0);
        if constexpr (F::KQ8) {
          sts64(qf + 256 * (KS * q + ch), pack_part(v.x * fq, v.y * fq, lo), pack_part(v.z * fq, v.w * fq, lo));
        } else {
          const float4 u = *reinterpret_cast<const float4*>(qp + D + c0);
          sts128(qf + 512 * (KS * q + ch), pack_part(v.x * fq, v.y * fq, lo), pack_part(v.z * fq, v.w * fq, lo),
                 pack_part(u.x * fs, u.y * fs, lo), pack_part(u.z * fs, u.w * fs, lo));
        }
      }
    }
    __syncwarp();
#pragma unroll
    for (int v = 0; v < NV; ++v) {
#pragma unroll
      for (int mt = 0; mt < KS; ++mt) oacc[v][mt][0] = oacc[v][mt][1] = oacc[v][mt][2] = oacc[v][mt][3] = 0.f;
    }
#pragma unroll
    for (int h = 0; h < NH; ++h) {
      m[h] = -INFINITY;
      l[h] = 0.f;
    }

    ntiles = t1 > t0 ? (t1 - t0 + 15) / 16 : 0;
    last_valid = t1 - t0 - 16 * (ntiles - 1);
    if (ntiles > 0) {
      c.page_ord = t0 / a.k.page_size;
      c.in_page = t0 - c.page_ord * a.k.page_size;
      set_page(c);
      prefetch_tiles(0, 0, kPrefetchTiles);
      // P' tiles: consecutive steps alternate between the two halves of the warp's P' block, so a
      // step's writes never meet the previous step's reads
      // (every step call uses buf, then flips it)
      uint32_t buf = 0;
      constexpr uint32_t kHalf = 256 * Shape<F, NQ>::NT * Shape<F, NQ>::NV;
      int tile = 0;
      if constexpr (Shape<F, NQ>::NT == 2) {
        // leading pairs of whole tiles, pipelined; the rest (at most two tiles, the last one
        // possibly ragged) runs below
        const int np = (last_valid == 16 ? ntiles : ntiles - 1) / 2;
        if (np > 0) {
          Cursor c1 = c;
          advance(c1);
          load_k<true>(kn[0], c, 16);
          load_k<true>(kn[1], c1, 16);
          load_v<true>(vn[0], c, 16);
          load_v<true>(vn[1], c1, 16);
          for (int pi = 0; pi < np; ++pi) {
            prefetch_tiles(tile, kPrefetchTiles, 2);
            const Cursor cur[2] = {c, c1};
            const bool more = pi + 1 < np;
            if (more || tile + 2 < ntiles) {
              c = c1;
              advance(c);  // tile + 2
            }
            if (more) {
              c1 = c;
              advance(c1);  // tile + 3
              const Cursor nx[2] = {c, c1};
              step_pipelined<true>(cur, nx, buf);
            } else {
              step_pipelined<false>(cur, cur, buf);
            }
            buf ^= kHalf;
            tile += 2;
          }
        }
      }
      for (; tile < ntiles; tile += 2) {
        prefetch_tiles(tile, kPrefetchTiles, 2);  // the two tiles that follow the ones already requested
        if (tile + 1 >= ntiles) {
          step_one(c, true, buf);
          break;
        }
        const bool last = tile + 2 >= ntiles;
        if constexpr (Shape<F, NQ>::NT == 2) {
          Cursor c1 = c;
          advance(c1);
          if (c.ok && c1.ok) {
            const Cursor two[2] = {c, c1};
            if (last && last_valid < 16) step_tiles<2, false>(two, last_valid, buf);
            else step_tiles<2, true>(two, 16, buf);
            buf ^= kHalf;
          } else {
            step_one(c, false, buf);
            buf ^= kHalf;
            step_one(c1, last, buf);
            buf ^= kHalf;
          }
          c = c1;
        } else {
          step_one(c, false, buf);
          buf ^= kHalf;
          advance(c);
          step_one(c, last, buf);
          buf ^= kHalf;
        }
        if (last) break;
        advance(c);
      }
    }

    // ---- partial of this work item: (m, l, acc) per query head ----
#pragma unroll
    for (int h = 0; h < NH; ++h) {
#pragma unroll
      for (int o = 4; o < 32; o <<= 1) l[h] += __shfl_xor_sync(kFull, l[h], o);
    }
    const float inv_lam = F::VQ8 ? 1.0f : 1.0f / k.tab.f16_scale[F::VQ8 ? 0 : F::WV - 1];
#pragma unroll
    for (int h = 0; h < NH; ++h) {
      const int head = t + 4 * h;
      if (head >= gcn) continue;
      float v[2 * KS];
#pragma unroll
      for (int mt = 0; mt < KS; ++mt) {
        if (HILO) {
          v[2 * mt] = (oacc[0][mt][0] + oacc[0][mt][1]) * inv_lam;
          v[2 * mt + 1] = (oacc[0][mt][2] + oacc[0][mt][3]) * inv_lam;
        } else {
          v[2 * mt] = oacc[h >> 1][mt][h & 1] * inv_lam;
          v[2 * mt + 1] = oacc[h >> 1][mt][2 + (h & 1)] * inv_lam;
        }
      }
      float* dst = k.partial + ((row0 + gof + head) * k.n_splits + split) * (D + 4);
      float4* dv = reinterpret_cast<float4*>(dst + 4 + g * (D / 8));
#pragma unroll
      for (int q = 0; q < D / 32; ++q) st_keep_v4(dv + q, make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]), pol_keep);
      if (g == 0) st_keep_v2(dst, make_float2(m[h] == -INFINITY ? -INFINITY : m[h] * kLn2, l[h]), pol_keep);
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

template <class F, int NQ>
__global__ void __launch_bounds__(Shape<F, NQ>::Threads, 1) attend_mma_kernel(DecodeLaunch k) {
  using L = Shape<F, NQ>;
  extern __shared__ __align__(16) unsigned char sm[];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  // ---- shared layout: the larger table on the first boundary of its size, the smaller one right
  // below it when there is room (both powers of two, so it is aligned to its own size), else right
  // above; warp blocks (two P' tiles, then the query fragments) from the start up to the smaller
  // table, the rest above the tables ----
  const uint32_t sbase = static_cast<uint32_t>(__cvta_generic_to_shared(sm));
  const uint32_t bofs = L::Big ? ((L::Big - (sbase & (L::Big - 1u))) & (L::Big - 1u)) : 0u;
  const bool small_below = bofs >= L::Small;
  const uint32_t sofs = small_below ? bofs - L::Small : bofs + L::Big;
  const uint32_t n_below = (small_below ? sofs : bofs) / (uint32_t)L::Block;
  const uint32_t above = bofs + L::Big + (small_below ? 0u : L::Small);
  const uint32_t kofs = F::KLut >= L::VLut ? bofs : sofs;
  const uint32_t vofs = F::KLut >= L::VLut ? sofs : bofs;
  const uint32_t wofs = (uint32_t)warp < n_below ? warp * (uint32_t)L::Block
                                                 : above + (warp - n_below) * (uint32_t)L::Block;
  if constexpr (!F::KQ8) {
    constexpr int W = F::WK, n = 1 << (2 * W), cm = (1 << W) - 1, im = (1 << (W - 1)) - 1;
    const float* cb = k.tab.centroids + (W - 2) * 8;
    const float lam = k.tab.f16_scale[W - 2];
    for (int i = tid; i < n * 8; i += L::Threads) {  // four lanes' copies per 16-byte store
      const int e = i >> 3, r = i & 7, c0 = e & cm, c1 = e >> W;
      const uint32_t x = h2_as_u32(__floats2half2_rn(lam * cb[c0 & im], lam * cb[c1 & im]));
      const uint32_t y = h2_as_u32(__floats2half2_rn((c0 >> (W - 1)) ? 1.f : -1.f, (c1 >> (W - 1)) ? 1.f : -1.f));
      *reinterpret_cast<uint4*>(sm + kofs + e * 256 + r * 16) = make_uint4(x, x, x, x);
      *reinterpret_cast<uint4*>(sm + kofs + e * 256 + 128 + r * 16) = make_uint4(y, y, y, y);
    }
  }
  if constexpr (L::DualV) {
    // entry e (a byte of codes): the pair in its low 2W bits at + 0, the pair in its high 2W bits
    // at + 128
    constexpr int W = F::WV, cm = (1 << W) - 1, pm = (1 << (2 * W)) - 1;
    const float* cb = k.tab.centroids + (W - 1) * 8;
    const float lam = k.tab.f16_scale[W - 1];
    for (int i = tid; i < 256 * 8; i += L::Threads) {
      const int e = i >> 3, r = i & 7, lo = e & pm, hi = e >> (8 - 2 * W);
      const uint32_t x = h2_as_u32(__floats2half2_rn(lam * cb[lo & cm], lam * cb[lo >> W]));
      const uint32_t y = h2_as_u32(__floats2half2_rn(lam * cb[hi & cm], lam * cb[hi >> W]));
      *reinterpret_cast<uint4*>(sm + vofs + e * 256 + r * 16) = make_uint4(x, x, x, x);
      *reinterpret_cast<uint4*>(sm + vofs + e * 256 + 128 + r * 16) = make_uint4(y, y, y, y);
    }
  } else if constexpr (!F::VQ8) {
    constexpr int W = F::WV, n = 1 << (2 * W), cm = (1 << W) - 1;
    const float* cb = k.tab.centroids + (W - 1) * 8;
    const float lam = k.tab.f16_scale[W - 1];
    for (int i = tid; i < n * 8; i += L::Threads) {
      const int e = i >> 3, r = i & 7;
      const uint32_t x = h2_as_u32(__floats2half2_rn(lam * cb[e & cm], lam * cb[e >> W]));
      *reinterpret_cast<uint4*>(sm + vofs + e * 128 + r * 16) = make_uint4(x, x, x, x);
    }
  }
  __syncthreads();
  pdl_wait();            // the query prologue (prepared queries, zeroed work counter) has completed
  pdl_launch_dependents();  // the combine may be scheduled as soon as SMs free up; it waits for this grid

  MmaWarp<F, NQ> w(k);
  w.init_lane(lane);
  w.ylk = (sbase + kofs) | ((uint32_t)lane << 2);
  w.ylv = (sbase + vofs) | ((uint32_t)lane << 2);
  const uint32_t ps = sbase + wofs;  // this warp's two P' tiles of 64 words, then its query fragments
  w.psw0 = ps + 4 * ps_word(2 * w.t, w.g);
  w.psw1 = ps + 4 * ps_word(2 * w.t + 1, w.g);
  w.psr = ps + 4 * ps_word(w.g, w.t);
  w.qf = ps + L::PsBytes + lane * (F::KQ8 ? 8 : 16);
  asm("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(w.pol));
  {
    uint64_t p_last, p_normal;
    asm("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p_last));
    asm("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(p_normal));
    w.pol_keep = k.keep_partials ? p_last : p_normal;
  }

  const DecodeArgs& a = k.a;
  const unsigned int n_items = (unsigned int)((long long)a.n_layers * a.batch * a.k.H * k.n_splits * k.g_halves);
  for (;;) {
    unsigned int item = 0;
    if (lane == 0) item = atomicAdd(k.counter, 1u);
    item = __shfl_sync(kFull, item, 0);
    if (item >= n_items) break;
    __syncwarp();  // the previous item's P' reads are done before this item's writes
    w.run_item(item);
  }
}

template <class F, int NQ>
cudaError_t launch_shape(const DecodeLaunch& k, long long items, int sm_count, cudaStream_t s) {
  using L = Shape<F, NQ>;
  long long grid = sm_count;  // one persistent CTA per SM
  if (items < grid * L::Warps) grid = (items + L::Warps - 1) / L::Warps;
  if (grid < 1) grid = 1;
  const cudaError_t e =
      cudaFuncSetAttribute(attend_mma_kernel<F, NQ>, cudaFuncAttributeMaxDynamicSharedMemorySize, L::Smem);
  if (e != cudaSuccess) return e;
  // a dependent of the query prologue: the tables are built while it runs
  return launch_pdl(attend_mma_kernel<F, NQ>, dim3((unsigned)grid), dim3(L::Threads), (size_t)L::Smem, s, k);
}

template <class F>
cudaError_t launch_mma(const DecodeLaunch& k, int sm_count, cudaStream_t s) {
  const long long items = (long long)k.a.n_layers * k.a.batch * k.a.k.H * k.n_splits * k.g_halves;
  if (items >= (1LL << 32)) return cudaErrorInvalidValue;
  if (k.g_cnt <= 4) return launch_shape<F, 1>(k, items, sm_count, s);
  if constexpr (F::D > 128) {
    return launch_shape<F, 2>(k, items, sm_count, s);
  } else {
    if (k.g_cnt <= 8) return launch_shape<F, 2>(k, items, sm_count, s);
    return launch_shape<F, 4>(k, items, sm_count, s);  // 9 to 16 heads: each tile dequantised once for all
  }
}

}  // namespace mmad
}  // namespace tq
