// Split-K decode attention over turbo K (QJL) and turbo-MSE V at head_dim 128, with the score
// products on the fifth-generation tensor cores (tcgen05, accumulators in tensor memory) and the
// value products on mma.sync.  Same work split, partials and combine as the split-K kernel of
// tq_decode_mma.cuh; a different engine for the scores.
//
// Why: with mma.sync every lane assembles A fragments of two tokens per k step from table
// lookups, and that operand assembly is most of the warp instructions of a tile.  Here thread i
// of a 128-thread group owns token i of the tile: one 8-byte table read per pair of coordinates
// gives the codebook pair lambda c[idx] and the QJL sign pair, and both go straight into tensor
// memory, interleaved, where they are the A operand (M = 128 tokens, K = 2d, one token per lane)
// of tcgen05.mma against the high / low fp16 parts of every query head's q' (codebook product,
// zeros at the sign elements) and S q' (QJL product, zeros at the codebook elements), the B
// operands in shared memory (N = 2 x heads).  One thread issues the 32 MMAs of a tile.  The value product contracts over tokens, which the token-major code layout
// does not give a tensor-core operand, so it stays on mma.sync m16n8k16 with fragment lookups.
//   score = n (c . q') + rnorm sqrt(pi/2)/d (sign . S q')    ("TurboQuant+ KV cache compression",
//   Stage 2: the QJL residual estimate; "TurboQuant+ deep dive", the decode path)
//
// Work: a group of four warps takes a work item = (layer x sequence, KV head, four consecutive
// splits) from an atomic counter; warp w runs split 4q + w, 32 tokens per tile in its own lane
// quarter of the tensor memory, and writes the partial (m, l, acc) of every query head and its
// split, exactly as the split-K kernel does.  The four warps share the tile's MMAs and meet at
// one named barrier per tile.  Three groups per CTA (two with 9 to 16 query heads), one CTA per
// SM; 512 columns of tensor memory hold each group's A (128 columns) and scores (2N).
// Per tile: K dequantisation into tensor memory; barrier; MMAs issued; the next tile's K loads;
// the previous tile's V products (overlapping the MMAs); this tile's V loads; wait for the MMAs;
// scores; online softmax (base 2, reference raised lazily, only when a score passes it by 2^8);
// Sparse V; P' into the warp's shared tile.  Every wait is bounded: one that runs out
// sets the status flag and ends the group's work.
#include "tq_decode_mma.cuh"
#include "tq_tc.cuh"

namespace tq {
namespace dtc {

using namespace wm;

// Kernel shape: turbo K code width WK (index bits + 1), turbo-MSE V code width WV, NQ = 1 (up to
// 4 query heads per KV head: P' as high / low fp16 parts), 2 (up to 8) or 4 (up to 16).
template <int WK_, int WV_, int NQ_>
struct Cfg {
  static constexpr int WK = WK_, WV = WV_, NQ = NQ_;
  using F = mmad::Fmt<128, WK, WV>;
  static constexpr int D = 128, KS = 8;
  static constexpr bool HILO = NQ == 1;
  static constexpr int GMAX = HILO ? 4 : 4 * NQ;
  static constexpr int NV = HILO ? 1 : NQ / 2;                // 8-column V products
  static constexpr int N = 2 * GMAX < 16 ? 16 : 2 * GMAX;     // score columns: high / low part per head
  static constexpr int Groups = NQ == 4 ? 2 : 3;
  static constexpr int Warps = 4 * Groups, Threads = 32 * Warps;
  static constexpr uint32_t GroupCols = 128 + 2 * N <= 160 ? 160u : 256u;
  static constexpr int KW = F::KPay / 4;                      // K payload words per token
  // Shared memory: the K table (entries of 2 x 4 bytes per lane, 256-byte stride) on a boundary
  // of its size, then the rest from the next boundary of RAlign: per group the two B operands
  // (1024-byte aligned), the V table (aligned to its size), per warp its P' tiles, barriers and
  // slots.
  static constexpr uint32_t KLut = 256u << (2 * WK), VLut = 128u << (2 * WV);
  static constexpr uint32_t BBytes = 2u * N * 512u;  // two operands of N rows x 256 f16
  static constexpr uint32_t PBytes = 2u * NV * 256u;
  static constexpr uint32_t RAlign = VLut > 1024u ? VLut : 1024u;
  static constexpr uint32_t oB = 0, oV = Groups * BBytes, oP = oV + VLut, oBar = oP + Warps * PBytes;
  static constexpr uint32_t oSlot = oBar + 8u * Groups, oItem = oSlot + 16u;
  static constexpr uint32_t RBytes = oItem + 8u * Groups;
  static constexpr uint32_t Need = (KLut - 16u) + KLut + (KLut < RAlign ? RAlign : 0u) + RBytes;
  // at least ~116 KB, so that a second CTA never shares the SM (and its tensor memory)
  static constexpr uint32_t Smem = Need > 118u * 1024u ? Need : 118u * 1024u;
  static_assert(Groups * GroupCols <= 512, "tensor memory");
  static_assert(BBytes % RAlign == 0, "V table alignment");
  static_assert(Smem <= 227u * 1024u, "shared memory");
  static_assert(KW % 4 == 0, "K rows of whole 16-byte words");
};

// V codes of one 16-token sub-tile in the fragment mapping of the V product: thread (g, t) holds
// the run of coordinates 16 g .. 16 g + 15 of tokens t, t + 8, t + 4, t + 12.
template <class F>
struct VSub {
  uint32_t w[4][F::VLoad];
};

__device__ __forceinline__ void sts16(uint32_t addr, __half h) {
  asm volatile("st.shared.u16 [%0], %1;" ::"r"(addr), "h"(*reinterpret_cast<unsigned short*>(&h)) : "memory");
}

__device__ __forceinline__ uint32_t pack_part(float x0, float x1, bool lo) {
  const __half2 hi = __floats2half2_rn(x0, x1);
  if (!lo) return h2_as_u32(hi);
  const float2 hf = __half22float2(hi);
  return h2_as_u32(__floats2half2_rn(x0 - hf.x, x1 - hf.y));
}

// First vector (in its layer) of the 16-token sub-tile at token `tok` of sequence b, KV head kvh.
// With a block table the page comes from it (an out-of-range entry is flagged and reads page 0).
__device__ __forceinline__ long long sub_vector(const DecodeLaunch& k, int b, int kvh, int page_ord, int in_page) {
  const DecodeArgs& a = k.a;
  long long page = b;
  if (a.block_table) {
    page = a.block_table[(long long)b * a.max_blocks_per_seq + page_ord];
    if (page < 0 || page >= a.k.num_pages) {
      atomicOr(k.tab.status, kFlagBlockTable);
      page = 0;
    }
  }
  return (page * a.k.H + kvh) * a.k.page_size + in_page;
}

template <int WK, int WV, int NQ>
__global__ void __launch_bounds__(Cfg<WK, WV, NQ>::Threads, 1) attend_tc_kernel(DecodeLaunch k) {
  using C = Cfg<WK, WV, NQ>;
  using F = typename C::F;
  constexpr int D = C::D, KS = C::KS, GMAX = C::GMAX, NV = C::NV, N = C::N, KW = C::KW;
  constexpr bool HILO = C::HILO;
  extern __shared__ __align__(16) unsigned char sm[];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int grp = warp >> 2, wq = warp & 3, gtid = tid & 127;
  const int g = lane >> 2, t = lane & 3;
  const uint32_t sbase = tc::smem_addr(sm);
  const uint32_t kofs = (C::KLut - (sbase & (C::KLut - 1u))) & (C::KLut - 1u);
  const uint32_t rofs = ((sbase + kofs + C::KLut + C::RAlign - 1u) & ~(C::RAlign - 1u)) - sbase;
  unsigned char* R = sm + rofs;
  uint64_t* bars = reinterpret_cast<uint64_t*>(R + C::oBar);
  uint64_t* bar = bars + grp;
  uint32_t* tslot = reinterpret_cast<uint32_t*>(R + C::oSlot);
  uint32_t* islot = reinterpret_cast<uint32_t*>(R + C::oItem) + 2 * grp;

  // ---- tables: K entry e (the codes of two coordinates) = {lambda c pair, sign pair} per lane;
  // V entry e = the f16 pair lambda c[e & m], lambda c[e >> WV] per lane ----
  {
    constexpr int W = WK, n = 1 << (2 * W), cm = (1 << W) - 1, im = (1 << (W - 1)) - 1;
    const float* cb = k.tab.centroids + (W - 2) * 8;
    const float lam = k.tab.f16_scale[W - 2];
    for (int i = tid; i < n * 32; i += C::Threads) {
      const int e = i >> 5, r = i & 31, c0 = e & cm, c1 = e >> W;
      const __half2 cv = __floats2half2_rn(lam * cb[c0 & im], lam * cb[c1 & im]);
      const __half2 sv = __floats2half2_rn((c0 >> (W - 1)) ? 1.f : -1.f, (c1 >> (W - 1)) ? 1.f : -1.f);
      *reinterpret_cast<uint2*>(sm + kofs + e * 256 + r * 8) = make_uint2(h2_as_u32(cv), h2_as_u32(sv));
    }
  }
  {
    constexpr int W = WV, n = 1 << (2 * W), cm = (1 << W) - 1;
    const float* cb = k.tab.centroids + (W - 1) * 8;
    const float lam = k.tab.f16_scale[W - 1];
    for (int i = tid; i < n * 32; i += C::Threads) {
      const int e = i >> 5, r = i & 31;
      *reinterpret_cast<uint32_t*>(R + C::oV + e * 128 + r * 4) =
          h2_as_u32(__floats2half2_rn(lam * cb[e & cm], lam * cb[e >> W]));
    }
  }
  if (warp == 0) tc::tmem_alloc(tslot, 512);
  if (tid < C::Groups) tc::mbar_init(bars + tid, 1);
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tslot;
  const uint32_t tA = tmem + grp * C::GroupCols;  // A: column 2p codebook pair p, 2p + 1 sign pair p
  const uint32_t tD = tA + 128;                   // scores: [0, N) codebook product, [N, 2N) QJL product
  const uint32_t lq = (uint32_t)(32 * wq) << 16;  // this warp's lane quarter
  const uint32_t ylk = (sbase + kofs) | ((uint32_t)lane << 3);
  const uint32_t ylv = (sbase + rofs + C::oV) | ((uint32_t)lane << 2);
  const uint32_t bB = sbase + rofs + C::oB + grp * C::BBytes;
  const uint32_t pbase = sbase + rofs + C::oP + warp * C::PBytes;
  // P' tile (sub-tile j, product v) at pbase + 256 (j NV + v): column c's 16 token slots in 32
  // bytes, the reader's two words (slot pairs of tokens t, t + 8 and t + 4, t + 12) adjacent
  const uint32_t prd = pbase + g * 32 + t * 8;
  const int u = lane & 15;
  const uint32_t pwr = pbase + (lane >> 4) * (NV * 256) + (u & 3) * 8 + ((u >> 2) & 1) * 4 + (u >> 3) * 2;
  const uint32_t idesc = tc::idesc_f16_f32(128, N);

  // V fragment mapping: the run of 16 W-bit codes at bit 16 g W of each row
  const int vw0 = (g * F::VBits) >> 5;
  const int vgo = 4 * vw0;
  const uint32_t vsh = (uint32_t)(g * F::VBits) & 31u;
  int vwo[F::VLoad];
#pragma unroll
  for (int j = 0; j < F::VLoad; ++j) vwo[j] = 4 * (min(vw0 + j, F::VPay / 4 - 1) - vw0);

  const DecodeArgs& a = k.a;
  const int H = a.k.H, G = k.G, Hq = a.n_q_heads, ST = k.split_tokens, ps = a.k.page_size;
  const int n_quads = (k.n_splits + 3) >> 2;
  const unsigned int n_items = (unsigned int)((long long)a.n_layers * a.batch * H * n_quads);
  const long long lv = (long long)a.k.num_pages * H * ps;  // vectors per layer
  const float fq = kLog2e / k.tab.f16_scale[WK - 2], fs = kLog2e * kSqrtHalfPi / (float)D;
  const float inv_lam_v = 1.0f / k.tab.f16_scale[WV - 1];
  const float tau = a.skip_threshold;
  const bool pf_k = ((reinterpret_cast<uintptr_t>(a.k.payload) | reinterpret_cast<uintptr_t>(a.v.payload)) & 15) == 0;
  uint64_t pol;
  asm("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  const int bid = 1 + grp;  // the group's named barrier
  uint32_t phase = 0;       // MMA completions this group has waited for
  bool ok = true;

  for (int it = 0;; ++it) {
    if (gtid == 0) islot[it & 1] = atomicAdd(k.counter, 1u);
    tc::bar_sync(bid, 128);
    const unsigned int item = islot[it & 1];
    if (item >= n_items) break;  // group-uniform

    const int quad = (int)(item % (unsigned)n_quads);
    const unsigned int rest = item / (unsigned)n_quads;
    const int kvh = (int)(rest % (unsigned)H);
    const int lb = (int)(rest / (unsigned)H);
    const int layer = k_layer_of(a, lb / a.batch), layer_v = v_layer_of(a, lb / a.batch);
    const int b = lb % a.batch;
    int len = a.seq_lens[b];
    if (len < 0) len = 0;
    if (len > a.max_ctx) {
      if (gtid == 0) atomicOr(k.tab.status, kFlagSeqLen);
      len = a.max_ctx;
    }
    const long long row0 = (long long)lb * Hq + (long long)kvh * G;
    const int split = 4 * quad + wq;
    const bool has_split = split < k.n_splits;
    const int t0 = split * ST;
    const int t1 = has_split ? max(t0, min(t0 + ST, len)) : t0;
    const int n_tiles = (min(max(len - 4 * quad * ST, 0), ST) + 31) >> 5;  // the quad's first split is its longest
    const unsigned char* kpl = a.k.payload + (long long)layer * lv * F::KPay;
    const unsigned char* khl = a.k.header + (long long)layer * lv * F::KHdr;
    const unsigned char* vpl = a.v.payload + (long long)layer_v * lv * F::VPay;
    const unsigned char* vhl = a.v.header + (long long)layer_v * lv * F::VHdr;

    // ---- B operands over the interleaved K of A (element 4p + e: codebook part of coordinate
    // 2p + e; 4p + 2 + e: its sign part): the codebook operand holds q' (with log2 e / lambda_K)
    // at the codebook elements and zeros at the sign elements, the QJL operand S q' (with
    // log2 e sqrt(pi/2) / d) the other way round; row 2h / 2h + 1 = high / low fp16 part of head
    // h.  128-byte swizzle, K-major, K quarters of 64 elements N x 128 bytes apart ----
    for (int i = gtid; i < 2 * N * 32; i += 128) {
      const int part = i / (N * 32), rr = (i >> 5) % N, c = i & 31, h = rr >> 1;
      const bool lo = rr & 1;
      uint4 v4 = make_uint4(0u, 0u, 0u, 0u);
      if (h < G) {
        const float4 x = *reinterpret_cast<const float4*>(k.qprep + (row0 + h) * 2 * D + part * D + 4 * c);
        const float f = part ? fs : fq;
        const uint32_t w0 = pack_part(x.x * f, x.y * f, lo), w1 = pack_part(x.z * f, x.w * f, lo);
        v4 = part ? make_uint4(0u, w0, 0u, w1) : make_uint4(w0, 0u, w1, 0u);
      }
      const uint32_t off = part * (N * 512) + (c >> 3) * (N * 128) + rr * 128 + (((c & 7) ^ (rr & 7)) << 4);
      sts128(bB + off, v4.x, v4.y, v4.z, v4.w);
    }
    tc::fence_async_smem();  // the first tile's barrier publishes them to the MMAs

    float oacc[NV][KS][4];
#pragma unroll
    for (int v = 0; v < NV; ++v) {
#pragma unroll
      for (int mt = 0; mt < KS; ++mt) oacc[v][mt][0] = oacc[v][mt][1] = oacc[v][mt][2] = oacc[v][mt][3] = 0.f;
    }
    float m[GMAX], l[GMAX];
#pragma unroll
    for (int h = 0; h < GMAX; ++h) {
      m[h] = -INFINITY;
      l[h] = 0.f;
    }

    // ---- sub-tile positions: cursor (page, offset) of the warp's next sub-tile to load, and of
    // the next one to request into L2 (from the second tile on, eight sub-tiles ahead) ----
    int c_ord = t0 / ps, c_in = t0 - (t0 / ps) * ps;
    auto advance = [&](int& ord, int& in) {
      in += 16;
      if (in >= ps) {
        in -= ps;
        ++ord;
      }
    };
    int f_ord = c_ord, f_in = c_in, f_tok = t0 + 32;
    advance(f_ord, f_in);
    advance(f_ord, f_in);
    // positions of the next tile's two sub-tiles: first vector in the layer (-1: none) and valid rows
    long long nvec[2];
    int nval[2];
    int ntok = t0;  // first token of the next tile
    auto next_positions = [&]() {
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int tb = ntok + 16 * j;
        nval[j] = min(max(t1 - tb, 0), 16);
        nvec[j] = nval[j] > 0 ? sub_vector(k, b, kvh, c_ord, c_in) : -1;
        advance(c_ord, c_in);
      }
      ntok += 32;
    };
    auto prefetch = [&]() {  // lane 0: the next two sub-tiles
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        if (lane == 0 && f_tok < t1) {
          const long long vec = sub_vector(k, b, kvh, f_ord, f_in);
          if (pf_k) {
            prefetch_l2(kpl + vec * F::KPay, 16 * F::KPay);
            prefetch_l2(vpl + vec * F::VPay, 16 * F::VPay);
          }
          const unsigned char* kh = khl + vec * F::KHdr;
          const unsigned char* vh = vhl + vec * F::VHdr;
          if (((reinterpret_cast<uintptr_t>(kh) | reinterpret_cast<uintptr_t>(vh)) & 15) == 0) {  // 16-byte starts
            prefetch_l2(kh, 16 * F::KHdr);
            prefetch_l2(vh, 16 * F::VHdr);
          }
        }
        advance(f_ord, f_in);
        f_tok += 16;
      }
    };
    // K row, K header and V norm of this lane's token of the next tile
    uint32_t kw[KW], khdr = 0, kvn = 0;
    bool kval = false;
    auto load_k = [&]() {
      const int j = lane >> 4;
      kval = u < nval[j];
      const long long vec = kval ? nvec[j] + u : 0;
      const unsigned char* kp = kval ? kpl + vec * F::KPay : a.k.payload;
      const unsigned char* kh = kval ? khl + vec * F::KHdr : a.k.header;
      const unsigned char* vh = kval ? vhl + vec * F::VHdr : a.v.header;
#pragma unroll
      for (int q = 0; q < KW; q += 4) {
        const uint4 x = ld_stream_v4(kp + 4 * q, pol);
        kw[q] = x.x; kw[q + 1] = x.y; kw[q + 2] = x.z; kw[q + 3] = x.w;
      }
      khdr = ld_stream_u32(kh, pol);
      kvn = ld_stream_u16(vh, pol);
    };
    // V codes of a tile's two sub-tiles at positions pv / pn (rows beyond the valid ones re-read
    // the last)
    auto load_v = [&](VSub<F> (&V)[2], const long long (&pv)[2], const int (&pn)[2]) {
      const int rows[4] = {t, t + 8, t + 4, t + 12};
#pragma unroll
      for (int j = 0; j < 2; ++j) {
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          const unsigned char* p =
              pn[j] > 0 ? vpl + (pv[j] + min(rows[r], pn[j] - 1)) * F::VPay + vgo : a.v.payload + vgo;
          if constexpr (F::VLoad == 1 || !F::VShift) {
            mmad::load_words<F::VLoad, F::VVec>(V[j].w[r], p, pol);
          } else {
#pragma unroll
            for (int q = 0; q < F::VLoad; ++q) V[j].w[r][q] = ld_stream_u32(p + vwo[q], pol);
          }
        }
      }
    };
    // V products of a tile whose P' is in the warp's tiles (sub-tiles without a kept weight skipped)
    auto v_products = [&](const VSub<F> (&V)[2], uint32_t skip) {
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        if (skip & (1u << j)) continue;  // warp-uniform
        uint2 bp[NV];
#pragma unroll
        for (int v = 0; v < NV; ++v) bp[v] = lds64_v(prd + 256 * (j * NV + v));
        constexpr int N2 = 2 * F::WV;
        uint32_t r[4][F::VRun];
#pragma unroll
        for (int q = 0; q < 4; ++q) mmad::make_run<F::VLoad, F::VRun, F::VShift>(V[j].w[q], r[q], vsh);
#pragma unroll
        for (int mt = 0; mt < KS; ++mt) {
          uint32_t e[4];
#pragma unroll
          for (int q = 0; q < 4; ++q) e[q] = lds32(mmad::run_addr<N2, 7>(r[q], 2 * mt * F::WV, ylv));
          // a0 / a1: slots 2t, 2t + 1 = tokens t, t + 8 at coordinates 16 g + 2 mt, + 1; a2 / a3:
          // tokens t + 4, t + 12
          const uint32_t a0 = __byte_perm(e[0], e[1], 0x5410), a1 = __byte_perm(e[0], e[1], 0x7632);
          const uint32_t a2 = __byte_perm(e[2], e[3], 0x5410), a3 = __byte_perm(e[2], e[3], 0x7632);
#pragma unroll
          for (int v = 0; v < NV; ++v) mma_16816(oacc[v][mt], a0, a1, a2, a3, bp[v].x, bp[v].y);
        }
      }
    };

    uint32_t skip_prev = 3u;  // sub-tiles of the previous tile without a kept weight
    // Tile i (its K in kw, its positions in nvec / nval): V holds tile i - 1's V codes, whose
    // products run here, and then receives tile i's.  False when a wait ran out (group-uniform).
    VSub<F> V[2];
    auto tile = [&](int i) -> bool {
      // 1. K of this tile into tensor memory: one table read per pair of coordinates lands in
      // two consecutive columns (codebook pair, sign pair)
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        uint32_t cs[16];
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const int p = 8 * c + q;  // coordinates 2p, 2p + 1
          uint32_t addr;
          if constexpr (WK == 4) addr = __byte_perm(kw[p >> 2], ylk, 0x7604u | ((uint32_t)(p & 3) << 4));
          else addr = mmad::run_addr<2 * WK, 8>(kw, 2 * WK * p, ylk);
          const uint2 e = lds64(addr);
          cs[2 * q] = e.x;
          cs[2 * q + 1] = e.y;
        }
        tc::tmem_st16(lq | (tA + 16 * c), cs);
      }
      const uint32_t hdr = khdr, vnorm = kvn;
      const bool val = kval;
      tc::tmem_wait_st();
      tc::fence_before_sync();
      tc::bar_sync(bid, 128);
      // 2. the score products (one thread)
      if (gtid == 0) {
        tc::fence_after_sync();
#pragma unroll
        for (int ks = 0; ks < 2 * KS; ++ks) {  // K = 256 interleaved elements, 16 per step
          const uint64_t db = tc::desc_sw128(bB + (ks >> 2) * (N * 128)) + (uint64_t)(2 * (ks & 3));
          tc::mma_f16_ts(tD, tA + 8 * ks, db, idesc, ks > 0);
          tc::mma_f16_ts(tD + N, tA + 8 * ks, db + (uint64_t)((N * 512) >> 4), idesc, ks > 0);
        }
        tc::commit(bar);
      }
      __syncwarp();
      // 3. the next tile's K; the previous tile's V products; this tile's V
      const long long pv[2] = {nvec[0], nvec[1]};
      const int pn[2] = {nval[0], nval[1]};
      if (i + 1 < n_tiles) {
        next_positions();
        load_k();
        prefetch();
      }
      if (i > 0) v_products(V, skip_prev);
      load_v(V, pv, pn);
      // 4. scores of this tile
      const bool done = tc::mbar_wait(bar, phase & 1u);
      ++phase;
      if (!tc::bar_sync_and(bid, 128, done)) return false;
      tc::fence_after_sync();
      float s[GMAX];
      {
        uint32_t sc[32];
        const float2 nr = __half22float2(u32_as_h2(hdr));  // norm, residual norm
        if constexpr (N == 16) {
          tc::tmem_ld32(lq | tD, sc);  // 16 codebook columns, then 16 QJL columns
#pragma unroll
          for (int h = 0; h < GMAX; ++h)
            s[h] = fmaf(nr.x, __uint_as_float(sc[2 * h]) + __uint_as_float(sc[2 * h + 1]),
                        nr.y * (__uint_as_float(sc[16 + 2 * h]) + __uint_as_float(sc[16 + 2 * h + 1])));
        } else {
          float cbs[GMAX];
          tc::tmem_ld32(lq | tD, sc);
#pragma unroll
          for (int h = 0; h < GMAX; ++h) cbs[h] = __uint_as_float(sc[2 * h]) + __uint_as_float(sc[2 * h + 1]);
          tc::tmem_ld32(lq | (tD + N), sc);
#pragma unroll
          for (int h = 0; h < GMAX; ++h)
            s[h] = fmaf(nr.x, cbs[h], nr.y * (__uint_as_float(sc[2 * h]) + __uint_as_float(sc[2 * h + 1])));
        }
      }
      // 5. online softmax: a head's reference is raised (to the warp's maximum) only when a score
      // passes it by 2^8; sums and accumulators are rescaled then
      bool need = false;
#pragma unroll
      for (int h = 0; h < GMAX; ++h) {
        if (!val || h >= G) s[h] = -INFINITY;
        need |= s[h] > m[h] + kLazyMax;
      }
      if (__any_sync(kFull, need)) {
        float al[GMAX];
#pragma unroll
        for (int h = 0; h < GMAX; ++h) {
          float mx = s[h];
#pragma unroll
          for (int o = 1; o < 32; o <<= 1) mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, o));
          const float mn = fmaxf(m[h], mx);
          al[h] = mn == -INFINITY ? 1.f : ex2(m[h] - mn);
          m[h] = mn;
          l[h] *= al[h];
        }
        // this thread's accumulator columns: 2t, 2t + 1 of product v
        if constexpr (HILO) {
          float f = al[0];
#pragma unroll
          for (int h = 1; h < GMAX; ++h) f = t == h ? al[h] : f;
#pragma unroll
          for (int mt = 0; mt < KS; ++mt) {
#pragma unroll
            for (int e = 0; e < 4; ++e) oacc[0][mt][e] *= f;
          }
        } else {
#pragma unroll
          for (int v = 0; v < NV; ++v) {
            float f0 = 1.f, f1 = 1.f;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              f0 = t == q ? al[8 * v + 2 * q] : f0;
              f1 = t == q ? al[8 * v + 2 * q + 1] : f1;
            }
#pragma unroll
            for (int mt = 0; mt < KS; ++mt) {
              oacc[v][mt][0] *= f0;
              oacc[v][mt][2] *= f0;
              oacc[v][mt][1] *= f1;
              oacc[v][mt][3] *= f1;
            }
          }
        }
      }
      float p[GMAX];
      bool any = false;
#pragma unroll
      for (int h = 0; h < GMAX; ++h) {
        p[h] = s[h] == -INFINITY ? 0.f : ex2(s[h] - m[h]);
        l[h] += p[h];
        if (tau > 0.f) p[h] = p[h] >= tau ? p[h] : 0.f;  // Sparse V
        any |= p[h] > 0.f;
      }
      const uint32_t bal = __ballot_sync(kFull, any);
      skip_prev = ((bal & 0xFFFFu) == 0u ? 1u : 0u) | ((bal >> 16) == 0u ? 2u : 0u);
      // 6. P' = weight * V norm into the warp's tiles (the previous tile's V products have read them)
      const float nv = __half2float(__ushort_as_half((unsigned short)vnorm));
      __syncwarp();
      if constexpr (HILO) {
#pragma unroll
        for (int h = 0; h < GMAX; ++h) {
          const float w = p[h] > 0.f ? p[h] * nv : 0.f;
          const __half hi = __float2half_rn(w);
          sts16(pwr + (2 * h) * 32, hi);
          sts16(pwr + (2 * h + 1) * 32, __float2half_rn(w - __half2float(hi)));
        }
      } else {
#pragma unroll
        for (int h = 0; h < GMAX; ++h) sts16(pwr + (h >> 3) * 256 + (h & 7) * 32, __float2half_rn(p[h] > 0.f ? p[h] * nv : 0.f));
      }
      __syncwarp();
      return true;
    };

    if (n_tiles > 0) {
      next_positions();
      load_k();
      prefetch();  // tiles 1 .. 4; then each tile requests the one four ahead of its loads
      prefetch();
      prefetch();
      prefetch();
      for (int i = 0; i < n_tiles && ok; ++i) ok = tile(i);
      if (ok) v_products(V, skip_prev);
    }
    if (!ok) break;  // group-uniform

    // ---- the partial of this warp's split: (m, l, acc) per query head ----
    if (has_split) {
#pragma unroll
      for (int h = 0; h < GMAX; ++h) {
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) l[h] += __shfl_xor_sync(kFull, l[h], o);
      }
#pragma unroll
      for (int e = 0; e < (HILO ? 1 : 2 * NV); ++e) {
        const int head = HILO ? t : 8 * (e >> 1) + 2 * t + (e & 1);
        if (head >= G) continue;
        float mh = m[0], lh = l[0];
#pragma unroll
        for (int h = 1; h < GMAX; ++h) {
          mh = head == h ? m[h] : mh;
          lh = head == h ? l[h] : lh;
        }
        float vals[2 * KS];
#pragma unroll
        for (int mt = 0; mt < KS; ++mt) {
          if constexpr (HILO) {
            vals[2 * mt] = (oacc[0][mt][0] + oacc[0][mt][1]) * inv_lam_v;
            vals[2 * mt + 1] = (oacc[0][mt][2] + oacc[0][mt][3]) * inv_lam_v;
          } else {
            vals[2 * mt] = oacc[e >> 1][mt][e & 1] * inv_lam_v;
            vals[2 * mt + 1] = oacc[e >> 1][mt][2 + (e & 1)] * inv_lam_v;
          }
        }
        float* dst = k.partial + ((row0 + head) * k.n_splits + split) * (D + 4);
        float4* dv = reinterpret_cast<float4*>(dst + 4 + g * (D / 8));
#pragma unroll
        for (int q = 0; q < D / 32; ++q) dv[q] = make_float4(vals[4 * q], vals[4 * q + 1], vals[4 * q + 2], vals[4 * q + 3]);
        if (g == 0) {
          dst[0] = mh == -INFINITY ? -INFINITY : mh * kLn2;
          dst[1] = lh;
        }
      }
    }
  }

  if (!ok && gtid == 0) {
    atomicOr(k.tab.status, kFlagTimeout);
    tc::mbar_wait(bar, (phase - 1u) & 1u, 1 << 10);  // the MMAs in flight, before the memory is freed
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(tmem, 512);
}

template <int WK, int WV, int NQ>
cudaError_t launch_tc(const DecodeLaunch& k, int sm_count, cudaStream_t s) {
  using C = Cfg<WK, WV, NQ>;
  const long long items = (long long)k.a.n_layers * k.a.batch * k.a.k.H * ((k.n_splits + 3) / 4);
  if (items >= (1LL << 32)) return cudaErrorInvalidValue;
  long long grid = sm_count;  // one persistent CTA per SM
  if (items < grid * C::Groups) grid = (items + C::Groups - 1) / C::Groups;
  if (grid < 1) grid = 1;
  const cudaError_t e =
      cudaFuncSetAttribute(attend_tc_kernel<WK, WV, NQ>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::Smem);
  if (e != cudaSuccess) return e;
  attend_tc_kernel<WK, WV, NQ><<<(unsigned)grid, C::Threads, C::Smem, s>>>(k);
  return cudaGetLastError();
}

template <int WK, int WV>
cudaError_t launch_heads(const DecodeLaunch& k, int sm_count, cudaStream_t s) {
  if (k.G <= 4) return launch_tc<WK, WV, 1>(k, sm_count, s);
  if (k.G <= 8) return launch_tc<WK, WV, 2>(k, sm_count, s);
  return launch_tc<WK, WV, 4>(k, sm_count, s);
}

}  // namespace dtc

bool tc_decode_has(int wk, int wv) { return wk >= 2 && wk <= 4 && wv >= 1 && wv <= 3; }

cudaError_t tc_decode_launch(const DecodeLaunch& k, int wk, int wv, int sm_count, cudaStream_t s) {
  using namespace dtc;
  if (!tc_decode_has(wk, wv) || k.G < 1 || k.G > 16) return cudaErrorInvalidValue;
#define TQ_TC_CASE(WK, WV) \
  case WK * 4 + WV:        \
    return launch_heads<WK, WV>(k, sm_count, s);
  switch (wk * 4 + wv) {
    TQ_TC_CASE(2, 1) TQ_TC_CASE(2, 2) TQ_TC_CASE(2, 3)
    TQ_TC_CASE(3, 1) TQ_TC_CASE(3, 2) TQ_TC_CASE(3, 3)
    TQ_TC_CASE(4, 1) TQ_TC_CASE(4, 2) TQ_TC_CASE(4, 3)
  }
#undef TQ_TC_CASE
  return cudaErrorInvalidValue;
}

}  // namespace tq
