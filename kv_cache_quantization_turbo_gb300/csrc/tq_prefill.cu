// Chunked-prefill attention over the compressed cache on fifth-generation tensor cores.
//
// A chunk of C new tokens at positions start .. start + C - 1 of one sequence, whose K and V are
// already in the compressed cache, attends causally to the cached tokens 0 .. its own position
// ("TurboQuant+: 3.8x compression ...", core content item 1: prefill over the quantised cache).
// Unlike a decode step, every K and V tile is used by many query rows, so the path is a dense
// contraction: the tiles are dequantised once into shared memory and the products run as
// tcgen05.mma with the accumulators in tensor memory.
//
// One CTA = 128 query rows of one KV head (row r = chunk token r / G, query head r % G of the
// KV head's group), three roles that run concurrently over the 64-key tiles (the warps of each
// listed at kThreads):
//   - row warps 0-3, one row per thread: the query as high and low fp16 parts of q' and S q'
//     (about 21 significant bits, with log2 e / lambda_K and log2 e sqrt(pi/2) / d folded in)
//     in tensor memory once, the A operand of the score products; per tile they read the row of
//     both products, form s_j = n_j S_cb + rnorm_j S_qjl (log2 units), mask keys after the
//     row's position, keep the online softmax (the running max raised lazily: the output in
//     tensor memory is rescaled only when the max passes the reference by 2^8) and write
//     P_j = 2^(s_j - m) |v_j| as fp16, the A operand of the value product;
//   - four producer warps: per tile, a thread dequantises half of one token: the codebook part
//     lambda_K c[idx] and the QJL sign part +-1 of K (turbo4: one table read per code byte) into
//     two K-major operand tiles [64 tokens x 128], V (lambda_V c_V[idx], one table read per pair of
//     coordinates) token-major into the MN-major B operand of the value product, and the
//     per-token norms; two tile buffers, so tile j + 1 is dequantised while tile j is in the
//     products and the softmax;
//   - one thread of the issuer warp: the score products S_cb = (q'_hi + q'_lo) K_cb^T and S_qjl =
//     (S q'_hi + S q'_lo) K_sign^T (M 128, N 64) of tile j + 1 as soon as its tiles are ready and
//     the row warps have read tile j's scores, then O += P V (M 128, N 128, K 64) of tile j.
// The roles meet only on mbarriers (tiles ready, scores done, scores read, P ready, values done);
// every wait is bounded, one that runs out sets the timeout bit and ends its role, and the others
// end by their own bounded waits.  The epilogue reads O, divides by the softmax sum and lambda_V,
// and applies diag(s) H (the inverse rotation) in registers.
#include <cuda_fp16.h>

#include "tq_device.cuh"
#include "tq_tc.cuh"

namespace tq {

__host__ __device__ constexpr float wm_log2e() { return 1.4426950408889634074f; }

namespace pf {

constexpr int D = 128;        // head_dim of this kernel
constexpr int M = 128;        // query rows per CTA
constexpr int NK = 64;        // keys per tile
// Warps: 0-7 rows (warp w: rows 32 (w % 4) .. + 31, keys 32 (w / 4) .. + 31 of each tile, so two
// warps per SM sub-partition share the softmax), 8-11 producers, 12 the MMA issuer.
constexpr int kRowWarps = 8, kProdWarps = 4, kIssuerWarp = 12;
constexpr int kThreads = 32 * 13;
__host__ __device__ constexpr int producer_index(int warp) {  // -1: not a producer
  return warp >= kRowWarps && warp < kRowWarps + kProdWarps ? warp - kRowWarps : -1;
}
constexpr uint32_t kTmemCols = 512;  // query parts [0, 256), S_cb [256, 320), S_qjl [320, 384), O [384, 512)
constexpr float kLazy = 8.0f;  // log2 units: rescale O when the row max passes the reference by this

// Byte offset of element (row r, column k) in a K-major operand tile of R rows whose K columns
// come in 64-element (128-byte) blocks with the 128-byte swizzle: block k / 64 at 128 R bytes,
// row r at 128 r, 16-byte chunk (k % 64) / 8 at position ((k % 64) / 8) ^ (r % 8).
template <int R>
__host__ __device__ constexpr int swz(int r, int k) {
  return (k >> 6) * (128 * R) + r * 128 + ((((k >> 3) & 7) ^ (r & 7)) << 4) + (k & 7) * 2;
}
// Byte offset of V element (token k, coordinate n) in the value product's B operand, MN-major with
// the 128-byte swizzle: 8-token groups of 1024 bytes (one 128-byte row per token, 64 coordinates,
// 16-byte chunk (n % 64) / 8 at position ((n % 64) / 8) ^ (k % 8)), coordinates 64 .. 127 8 KB on.
__host__ __device__ constexpr int swz_v(int k, int n) {
  return (n >> 6) * 8192 + (k >> 3) * 1024 + (k & 7) * 128 + ((((n >> 3) & 7) ^ (k & 7)) << 4) + (n & 7) * 2;
}
// Start offset of K step ks (16 columns) of such a tile.
template <int R>
__host__ __device__ constexpr uint32_t kstep(int ks) {
  return (uint32_t)((ks >> 2) * (128 * R) + (ks & 3) * 32);
}

constexpr int NB = 3;  // K / V tile buffers (P: two)
struct Smem {  // byte offsets from a 1024-byte boundary; [NB] = the K / V tile buffers
  static constexpr int kcb = 0;                       // [NB][64 x 128]
  static constexpr int ksg = kcb + NB * NK * D * 2;   // [NB][64 x 128]
  static constexpr int vt = ksg + NB * NK * D * 2;    // [NB][64 tokens x 128], MN-major (swz_v)
  static constexpr int p = vt + NB * D * NK * 2;      // [2][128 x 64]
  static constexpr int hdr = p + 2 * M * NK * 2;      // [NB] float kn[64], kr[64], vn[64]
  static constexpr int tab = hdr + NB * 3 * NK * 4;   // fp16 cb_k[8], cb_v[8]
  static constexpr int kbt = tab + 32;                // turbo4 K: uint2 [256] per code byte: codebook pair, sign pair
  static constexpr int vpt = kbt + 256 * 8;           // V: f16 pair per code pair (2 W_V bits) and lane: [64][32] words
  static constexpr int xch = vpt + 64 * 32 * 4;       // float [2][128]: half-tile row maxima, then half sums
  static constexpr int inval = xch + 2 * M * 4;       // uint32 [NB][4]: a producer warp's tile holds keys that are not there
  static constexpr int bar = inval + 16 * NB;         // mbarriers: kv_full[NB], s_done, s_free, p_full[2], pv_done[NB]
  static constexpr int slot = bar + 10 * 8;           // tensor-memory address
  static constexpr int total = slot + 16;
  static constexpr int alloc = total + 1024;          // room to align the base
};
static_assert(Smem::alloc <= 227 * 1024, "shared memory");

struct Args {
  DevView k, v;
  DevTables tab;
  int layer, seq;
  const int32_t* block_table;  // logical page -> physical page of the sequence, or null (page = seq)
  int max_blocks;
  int start, n_tokens, n_q_heads, G;
  const float* qprep;  // [n_tokens * n_q_heads][2 D]: q' (softmax scale folded in), then S q'
  float* out;          // [n_tokens][n_q_heads][D]
  float fq, fs;        // log2 e / lambda_K; log2 e sqrt(pi/2) / D
  float inv_lam_v;     // 1 / lambda_V
};

__device__ __forceinline__ uint32_t pack_h2(float a, float b) {
  const __half2 h = __floats2half2_rn(a, b);
  return *reinterpret_cast<const uint32_t*>(&h);
}
__device__ __forceinline__ float lo_part(float x) { return x - __half2float(__float2half_rn(x)); }
__device__ __forceinline__ float fast_ex2(float x) {  // 2^x; -inf -> 0
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Code of coordinate c (compile-time after unrolling) in the little-endian stream w of W-bit codes.
template <int W, int NW>
__device__ __forceinline__ uint32_t code_at(const uint32_t (&w)[NW], int c) {
  const int bit = W * c, i = bit >> 5, off = bit & 31;
  uint32_t x = w[i] >> off;
  if (off + W > 32) x |= w[i + 1 < NW ? i + 1 : i] << (32 - off);
  return x & ((1u << W) - 1u);
}

// True if the phase of the given parity of the mbarrier has completed (a non-blocking test).
__device__ __forceinline__ bool test_wait(uint64_t* bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}\n"
      : "=r"(done)
      : "r"(tc::smem_addr(bar)), "r"(parity)
      : "memory");
  return done != 0;
}

// The four score products of one K step (16 coordinates): the codebook accumulator d_cb += (q'_hi +
// q'_lo) K_cb and the QJL accumulator d_qj += (S q'_hi + S q'_lo) K_sign, A from tensor memory, B
// from the shared-memory descriptors {b_cb_lo, b_hi} and {b_sg_lo, b_hi}; acc = 0 starts both sums.
__device__ __forceinline__ void mma_kstep(uint32_t d_cb, uint32_t d_qj, uint32_t a_hi, uint32_t a_lo, uint32_t a_shi,
                                          uint32_t a_slo, uint32_t b_cb_lo, uint32_t b_sg_lo, uint32_t b_hi,
                                          uint32_t idesc, bool acc) {
  asm volatile(
      "{\n\t.reg .pred p, t;\n\t.reg .b64 bc, bs;\n\t"
      "setp.ne.b32 p, %10, 0;\n\tsetp.eq.b32 t, %10, %10;\n\t"
      "mov.b64 bc, {%6, %8};\n\tmov.b64 bs, {%7, %8};\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%2], bc, %9, p;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%3], bc, %9, t;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%1], [%4], bs, %9, p;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%1], [%5], bs, %9, t;\n\t}\n" ::"r"(d_cb),
      "r"(d_qj), "r"(a_hi), "r"(a_lo), "r"(a_shi), "r"(a_slo), "r"(b_cb_lo), "r"(b_sg_lo), "r"(b_hi), "r"(idesc),
      "r"((uint32_t)acc));
}

// One arrival per warp after the whole warp's shared-memory stores: made visible to the tensor
// core, then lane 0 arrives.
__device__ __forceinline__ void warp_arrive_smem(uint64_t* bar, int lane) {
  tc::fence_async_smem();
  __syncwarp();
  if (lane == 0) tc::mbar_arrive(bar);
}

template <int WK, int WV>  // K code width (turbo K: index bits + 1), V code width (turbo-MSE: index bits)
__global__ void __launch_bounds__(kThreads, 1) prefill_kernel(const __grid_constant__ Args a) {
  constexpr int BK = WK - 1;  // K index bits; bit BK of a K code is the QJL sign
  extern __shared__ __align__(16) unsigned char smem_raw[];
  unsigned char* sm = smem_raw + ((1024u - (tc::smem_addr(smem_raw) & 1023u)) & 1023u);
  const uint32_t sb = tc::smem_addr(sm);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  __half* cbk = reinterpret_cast<__half*>(sm + Smem::tab);
  __half* cbv = cbk + 8;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + Smem::bar);
  uint64_t* kv_full = bars;       // [NB] K / V tile buffer b dequantised (4 producer warps)
  uint64_t* s_done = bars + 3;    // the score products of a tile completed (commit)
  uint64_t* s_free = bars + 4;    // the row warps have read a tile's scores (8 row warps)
  uint64_t* p_full = bars + 5;    // [2] P buffer b written (8 row warps)
  uint64_t* pv_done = bars + 7;   // [NB] the value product of the tile in K / V buffer b completed (commit)
  uint32_t* slot = reinterpret_cast<uint32_t*>(sm + Smem::slot);

  const int kvh = blockIdx.y, G = a.G, Hq = a.n_q_heads;
  const int row0 = blockIdx.x * M;  // first row of this CTA in the KV head's rows (token i, head g) = i G + g
  if (warp == 0) {
    tc::tmem_alloc(slot, kTmemCols);
    if (lane == 0) {
      tc::mbar_init(kv_full, kProdWarps);
      tc::mbar_init(kv_full + 1, kProdWarps);
      tc::mbar_init(kv_full + 2, kProdWarps);
      tc::mbar_init(s_done, 1);
      tc::mbar_init(s_free, kRowWarps);  // one arrival per row warp (each reads half of the scores)
      tc::mbar_init(p_full, kRowWarps);
      tc::mbar_init(p_full + 1, kRowWarps);
      tc::mbar_init(pv_done, 1);
      tc::mbar_init(pv_done + 1, 1);
      tc::mbar_init(pv_done + 2, 1);
    }
  }
  if (tid < 8) {
    cbk[tid] = __float2half_rn(tid < (1 << BK) ? a.tab.f16_scale[BK - 1] * a.tab.centroids[(BK - 1) * 8 + tid] : 0.f);
    cbv[tid] = __float2half_rn(tid < (1 << WV) ? a.tab.f16_scale[WV - 1] * a.tab.centroids[(WV - 1) * 8 + tid] : 0.f);
  }
  if constexpr (WK == 4) {  // a byte of turbo4 K codes = two coordinates: their codebook pair and sign pair
    const float lam = a.tab.f16_scale[BK - 1];
    const float* cb = a.tab.centroids + (BK - 1) * 8;
    for (int b = tid; b < 256; b += kThreads) {
      const __half2 c2 = __floats2half2_rn(lam * cb[b & 7], lam * cb[(b >> 4) & 7]);
      const __half2 s2 = __floats2half2_rn((b & 8) ? 1.f : -1.f, (b & 128) ? 1.f : -1.f);
      *reinterpret_cast<uint2*>(sm + Smem::kbt + 8 * b) =
          make_uint2(*reinterpret_cast<const uint32_t*>(&c2), *reinterpret_cast<const uint32_t*>(&s2));
    }
  }
  {  // V pair table, replicated per lane: entry e = the code pair (low W_V bits: the first coordinate)
    constexpr int npair = 1 << (2 * WV), cm = (1 << WV) - 1;
    const float lam = a.tab.f16_scale[WV - 1];
    const float* cb = a.tab.centroids + (WV - 1) * 8;
    for (int i = tid; i < npair * 32; i += kThreads) {
      const int e = i >> 5;
      *reinterpret_cast<uint32_t*>(sm + Smem::vpt + 4 * i) = pack_h2(lam * cb[e & cm], lam * cb[e >> WV]);
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *slot;
  const uint32_t t_q = tmem, t_cb = tmem + 256, t_qj = tmem + 320, t_o = tmem + 384;
  const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;  // a row warp's tensor-memory lane quarter

  // ---- the query parts into tensor memory (row warps): columns 64 p .. 64 p + 63 of part p =
  // q'_hi, q'_lo, (S q')_hi, (S q')_lo, two f16 coordinates per column ----
  const bool row_warp = warp < kRowWarps;
  const int r = tid & (M - 1);
  const int rho = row0 + r, ti = rho / G, gi = rho - ti * G;
  const bool row_ok = row_warp && ti < a.n_tokens;
  const int pos = a.start + ti;  // this row's position: it attends to keys 0 .. pos
  if (row_warp) {
    const float* qp = a.qprep + ((long long)ti * Hq + kvh * G + gi) * 2 * D;
    {
      const int part = warp >> 2;  // warps 0-3: q'; 4-7: S q'
      const float f = part ? a.fs : a.fq;
#pragma unroll 1
      for (int c32 = 0; c32 < 2; ++c32) {  // coordinates 64 c32 .. 64 c32 + 63
        uint32_t hi[32], lo[32];
#pragma unroll
        for (int e4 = 0; e4 < 16; ++e4) {
          float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
          if (row_ok) x = *reinterpret_cast<const float4*>(qp + part * D + 64 * c32 + 4 * e4);
          x.x *= f; x.y *= f; x.z *= f; x.w *= f;
          hi[2 * e4] = pack_h2(x.x, x.y);
          hi[2 * e4 + 1] = pack_h2(x.z, x.w);
          lo[2 * e4] = pack_h2(lo_part(x.x), lo_part(x.y));
          lo[2 * e4 + 1] = pack_h2(lo_part(x.z), lo_part(x.w));
        }
        tc::tmem_st32(t_q + lane_base + 128 * part + 32 * c32, hi);
        tc::tmem_st32(t_q + lane_base + 128 * part + 64 + 32 * c32, lo);
      }
    }
    tc::tmem_wait_st();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();

  // keys this CTA reads: up to the last row's position; keys beyond the chunk are never attended
  const int last_row = min(row0 + M, a.n_tokens * G) - 1;
  const int n_keys = a.start + last_row / G + 1;
  const int n_tiles = (n_keys + NK - 1) / NK;
  const int first_pos = a.start + row0 / G;  // the smallest position of the CTA's rows
  const DevView& K = a.k;
  const DevView& V = a.v;
  const long long vec_layer = (long long)K.num_pages * K.H * K.page_size;
  bool ok = true;  // every bounded wait of this thread's role completed
  float m = -INFINITY, l = 0.f;

  if (producer_index(warp) >= 0) {
    // ================= producers: dequantise tile jt into buffer jt % 2 =================
    const int ptid = 32 * producer_index(warp) + lane;
    const int tt = ptid & (NK - 1), qh = ptid >> 6;  // token tt of the tile, coordinates 64 qh ..
    constexpr int NWK = 2 * WK, NWV = 2 * WV;        // 32-bit words of this thread's 64 codes
    // this thread's codes and norms of one tile, loaded a tile ahead of their dequantisation
    struct Codes {
      uint32_t wk[NWK], wv[NWV];
      __half n, rn, nv;
      bool valid;
    };
    auto load_codes = [&](int jt, Codes& c) {
      const int j = jt * NK + tt;
      c.valid = j < n_keys;
      long long vec = 0;
      if (c.valid) {
        long long page = a.seq;
        const int lp = j / K.page_size;
        if (a.block_table) {
          page = lp < a.max_blocks ? a.block_table[lp] : -1;
          if (page < 0 || page >= K.num_pages) {
            if (qh == 0) atomicOr(a.tab.status, kFlagBlockTable);
            c.valid = false;
          }
        }
        vec = (long long)a.layer * vec_layer + (page * K.H + kvh) * K.page_size + (j - lp * K.page_size);
      }
      if (c.valid) {
        const uint32_t* pk = reinterpret_cast<const uint32_t*>(K.payload + vec * K.pay_bytes) + qh * NWK;
        const uint32_t* pv = reinterpret_cast<const uint32_t*>(V.payload + vec * V.pay_bytes) + qh * NWV;
#pragma unroll
        for (int i = 0; i < NWK; ++i) c.wk[i] = __ldg(pk + i);
#pragma unroll
        for (int i = 0; i < NWV; ++i) c.wv[i] = __ldg(pv + i);
        const __half* hk = reinterpret_cast<const __half*>(K.header + vec * K.hdr_bytes);
        c.n = hk[0];
        c.rn = hk[1];
        c.nv = *reinterpret_cast<const __half*>(V.header + vec * V.hdr_bytes);
      } else {
#pragma unroll
        for (int i = 0; i < NWK; ++i) c.wk[i] = 0u;
#pragma unroll
        for (int i = 0; i < NWV; ++i) c.wv[i] = 0u;
        c.n = c.rn = c.nv = __float2half_rn(0.f);
      }
    };
    Codes cur, nxt;
    if (n_tiles > 0) load_codes(0, cur);
    for (int jt = 0; jt < n_tiles && ok; ++jt) {
      const int bf = jt % NB;
      if (jt + 1 < n_tiles) load_codes(jt + 1, nxt);  // in flight while this tile is dequantised
      if (jt >= NB) ok = tc::mbar_wait(pv_done + bf, (uint32_t)(jt / NB - 1) & 1u);  // buffer read by tile jt - NB
      if (!ok) break;
      tc::fence_after_sync();
      unsigned char* kcb_b = sm + Smem::kcb + bf * NK * D * 2;
      unsigned char* ksg_b = sm + Smem::ksg + bf * NK * D * 2;
      unsigned char* vt_b = sm + Smem::vt + bf * D * NK * 2;
      float* kn_s = reinterpret_cast<float*>(sm + Smem::hdr) + bf * 3 * NK;
      const bool valid = cur.valid;
      const uint32_t (&wk)[NWK] = cur.wk;
      const uint32_t (&wv)[NWV] = cur.wv;
      const __half hz = __float2half_rn(0.f), hp1 = __float2half_rn(1.f), hm1 = __float2half_rn(-1.f);
#pragma unroll
      for (int c8 = 0; c8 < 8; ++c8) {  // coordinates 64 qh + 8 c8 .. + 7
        uint4 kcb, ksg;
        if constexpr (WK == 4) {  // one table read per code byte (two coordinates)
          uint2 e[4];
#pragma unroll
          for (int b = 0; b < 4; ++b) e[b] = *reinterpret_cast<const uint2*>(sm + Smem::kbt + 8 * ((wk[c8] >> (8 * b)) & 255u));
          kcb = make_uint4(e[0].x, e[1].x, e[2].x, e[3].x);
          ksg = make_uint4(e[0].y, e[1].y, e[2].y, e[3].y);
          if (!valid) kcb = ksg = make_uint4(0u, 0u, 0u, 0u);
        } else {
          __half cbv8[8], sgv8[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const uint32_t code = code_at<WK, NWK>(wk, 8 * c8 + e);
            cbv8[e] = valid ? cbk[code & ((1u << BK) - 1u)] : hz;
            sgv8[e] = valid ? (((code >> BK) & 1u) ? hp1 : hm1) : hz;
          }
          kcb = *reinterpret_cast<const uint4*>(cbv8);
          ksg = *reinterpret_cast<const uint4*>(sgv8);
        }
        const int o = swz<NK>(tt, 64 * qh + 8 * c8);
        *reinterpret_cast<uint4*>(kcb_b + o) = kcb;
        *reinterpret_cast<uint4*>(ksg_b + o) = ksg;
        uint32_t vp[4];
#pragma unroll
        for (int e2 = 0; e2 < 4; ++e2) {  // coordinate pairs: one table read each
          const uint32_t pc = code_at<2 * WV, NWV>(wv, 4 * c8 + e2);
          vp[e2] = *reinterpret_cast<const uint32_t*>(sm + Smem::vpt + 128 * pc + 4 * lane);
        }
        if (!valid) vp[0] = vp[1] = vp[2] = vp[3] = 0u;
        *reinterpret_cast<uint4*>(vt_b + swz_v(tt, 64 * qh + 8 * c8)) = make_uint4(vp[0], vp[1], vp[2], vp[3]);
      }
      {
        const uint32_t any_invalid = __ballot_sync(kFull, !valid);
        if (lane == 0)
          reinterpret_cast<uint32_t*>(sm + Smem::inval)[4 * bf + producer_index(warp)] = any_invalid != 0u;
      }
      if (qh == 0) {
        kn_s[tt] = valid ? __half2float(cur.n) : NAN;  // NaN marks a key that is not there (masked by the row warps)
        kn_s[NK + tt] = __half2float(cur.rn);
        kn_s[2 * NK + tt] = __half2float(cur.nv);
      }
      warp_arrive_smem(kv_full + bf, lane);
      cur = nxt;
    }
  } else if (warp == kIssuerWarp) {
    // ================= MMA issue (one thread) =================
    // Whichever is ready first: the value product of the oldest scored tile (it frees a P and a K / V
    // buffer), else the score products of the next tile (its tiles dequantised, the previous scores
    // read).  Polls are non-blocking; their total is bounded (about a second).
    if (lane == 0) {
      constexpr uint32_t id64 = tc::idesc_f16_f32(M, NK);
      constexpr uint32_t id128v = tc::idesc_f16_f32(M, D) | (1u << 16);  // B (V) MN-major
      const uint32_t kDescHi = (uint32_t)(tc::desc_sw128(0) >> 32);  // a 128-byte-swizzle K-major descriptor's high word
      int ns = 0, np = 0;  // score / value products issued
      long long idle = 0;
      while (np < n_tiles) {
        bool did = false;
        if (np < ns && test_wait(p_full + (np & 1), (uint32_t)(np >> 1) & 1u)) {  // O += P V of tile np
          tc::fence_after_sync();
          const uint64_t dp = tc::desc_sw128(sb + Smem::p + (np & 1) * M * NK * 2);
          const uint64_t dv = tc::desc_sw128_mn(sb + Smem::vt + (np % NB) * D * NK * 2, 8192);
#pragma unroll
          for (int ks = 0; ks < NK / 16; ++ks)  // 16 tokens = two 1024-byte groups of V
            tc::mma_f16(t_o, dp + (kstep<M>(ks) >> 4), dv + (uint64_t)(ks * (2048 >> 4)), id128v, np > 0 || ks > 0);
          tc::commit(pv_done + np % NB);
          ++np;
          did = true;
        } else if (ns < n_tiles && test_wait(kv_full + ns % NB, (uint32_t)(ns / NB) & 1u) &&
                   (ns == 0 || test_wait(s_free, (uint32_t)(ns - 1) & 1u))) {
          // S_cb = (q'_hi + q'_lo) K_cb^T, S_qjl = (S q'_hi + S q'_lo) K_sign^T: one instruction block per
          // k step, the operand descriptors' low words stepped in 32 bits
          tc::fence_after_sync();
          const uint32_t lcb = (uint32_t)tc::desc_sw128(sb + Smem::kcb + (ns % NB) * NK * D * 2);
          const uint32_t lsg = (uint32_t)tc::desc_sw128(sb + Smem::ksg + (ns % NB) * NK * D * 2);
#pragma unroll
          for (int ks = 0; ks < D / 16; ++ks) {
            const uint32_t kb = kstep<NK>(ks) >> 4;
            mma_kstep(t_cb, t_qj, t_q + 8 * ks, t_q + 64 + 8 * ks, t_q + 128 + 8 * ks, t_q + 192 + 8 * ks, lcb + kb,
                      lsg + kb, kDescHi, id64, ks > 0);
          }
          tc::commit(s_done);
          ++ns;
          did = true;
        }
        if (did) {
          idle = 0;
        } else {
          if (++idle > (1 << 24)) {  // about a second of polls with nothing to issue
            ok = false;
            break;
          }
          __nanosleep(32);
        }
      }
      if (!ok) {  // bounded waits for the products still in flight before the tensor memory is freed
        if (ns > 0) tc::mbar_wait(s_done, (uint32_t)(ns - 1) & 1u, 1 << 10);
        if (np > 0) tc::mbar_wait(pv_done + (np - 1) % NB, (uint32_t)((np - 1) / NB) & 1u, 1 << 10);
      }
    }
    __syncwarp();
  } else if (row_warp) {
    // ================= row warps: scores, online softmax, P =================
    // warp w and w + 4 hold the same rows (the same tensor-memory lanes) and split each tile's keys;
    // they meet on named barrier 1 + w % 4, and every wait's outcome is made the pair's before
    // either of them can leave the loop
    const int kh = warp >> 2;
    const int pair_bar = 1 + (warp & 3);
    float* xch = reinterpret_cast<float*>(sm + Smem::xch);
    for (int jt = 0; jt < n_tiles && ok; ++jt) {
      const int bf = jt % NB, bp = jt & 1;  // K / V buffer, P buffer
      bool w_ok = tc::mbar_wait(s_done, (uint32_t)jt & 1u);
      if (w_ok) w_ok = tc::mbar_wait(kv_full + bf, (uint32_t)(jt / NB) & 1u);  // (complete: the tile's norms)
      ok = tc::bar_sync_and(pair_bar, 64, w_ok);
      if (!ok) break;
      tc::fence_after_sync();
      const float* kn_s = reinterpret_cast<const float*>(sm + Smem::hdr) + bf * 3 * NK + 32 * kh;
      const float* kr_s = kn_s + NK;
      const float* vn_s = kn_s + 2 * NK;
      float s[32];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        uint32_t vcb[16], vq[16];
        tc::tmem_ld16_nw(t_cb + lane_base + 32 * kh + 16 * h, vcb);
        tc::tmem_ld16_nw(t_qj + lane_base + 32 * kh + 16 * h, vq);
        tc::tmem_wait_ld();
        if (h == 1) {
          tc::fence_before_sync();
          __syncwarp();
          if (lane == 0) tc::mbar_arrive(s_free);  // this warp's half of the tile's scores is read
        }
#pragma unroll
        for (int e = 0; e < 16; ++e)
          s[16 * h + e] = fmaf(kn_s[16 * h + e], __uint_as_float(vcb[e]), kr_s[16 * h + e] * __uint_as_float(vq[e]));
      }
      // masks (keys after the row's position, keys that are not there) only where the tile reaches
      // past the first row's position or holds such keys; rows past the chunk are never stored
      const uint4 inv = *reinterpret_cast<const uint4*>(sm + Smem::inval + 16 * bf);
      const bool full = jt * NK + NK - 1 <= first_pos && (inv.x | inv.y | inv.z | inv.w) == 0u;
      if (!full) {
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          const bool keep = !isnan(kn_s[e]) && jt * NK + 32 * kh + e <= pos;
          s[e] = keep ? s[e] : -INFINITY;
        }
      }
      float mx[4];
#pragma unroll
      for (int q = 0; q < 4; ++q)
        mx[q] = fmaxf(fmaxf(fmaxf(s[q], s[4 + q]), fmaxf(s[8 + q], s[12 + q])),
                      fmaxf(fmaxf(s[16 + q], s[20 + q]), fmaxf(s[24 + q], s[28 + q])));
      xch[kh * M + r] = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
      tc::bar_sync(pair_bar, 64);
      const float mt = fmaxf(xch[r], xch[M + r]);  // the row's maximum over the tile (the same in both warps)
      // Raise the reference when a row's max passes it by 2^kLazy.  The tensor-memory loads and
      // stores are warp-collective, so the decision is the warp's (the same in both warps of the
      // rows): every row raises its reference to its running max (a factor of 1 where that changes
      // nothing), rescales its half of l and its half of the O row, once the value products so
      // far have completed.
      if (__any_sync(kFull, mt > m + kLazy)) {
        const float mn = fmaxf(m, mt);
        const float al = mn == -INFINITY ? 1.f : (m == -INFINITY ? 0.f : exp2f(m - mn));
        l *= al;
        if (jt > 0) {
          w_ok = tc::mbar_wait(pv_done + (jt - 1) % NB, (uint32_t)((jt - 1) / NB) & 1u);
          ok = tc::bar_sync_and(pair_bar, 64, w_ok);
          if (!ok) break;
          tc::fence_after_sync();
#pragma unroll 1
          for (int c32 = 0; c32 < 2; ++c32) {
            uint32_t ov[32];
            tc::tmem_ld32(t_o + lane_base + 64 * kh + 32 * c32, ov);
#pragma unroll
            for (int e = 0; e < 32; ++e) ov[e] = __float_as_uint(__uint_as_float(ov[e]) * al);
            tc::tmem_st32(t_o + lane_base + 64 * kh + 32 * c32, ov);
          }
          tc::tmem_wait_st();
          tc::fence_before_sync();
        }
        m = mn;
      }
      // P into buffer bp once the value product of tile jt - 2 has read it
      if (jt >= 2) {
        w_ok = tc::mbar_wait(pv_done + (jt - 2) % NB, (uint32_t)((jt - 2) / NB) & 1u);
        ok = tc::bar_sync_and(pair_bar, 64, w_ok);
        if (!ok) break;
      }
      unsigned char* p_b = sm + Smem::p + bp * M * NK * 2;
      float ls[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int c8 = 0; c8 < 4; ++c8) {
        uint32_t pk[4];
#pragma unroll
        for (int e2 = 0; e2 < 4; ++e2) {
          const int j0 = 8 * c8 + 2 * e2;
          const float p0 = s[j0] == -INFINITY ? 0.f : fast_ex2(s[j0] - m);
          const float p1 = s[j0 + 1] == -INFINITY ? 0.f : fast_ex2(s[j0 + 1] - m);
          ls[e2] += p0 + p1;
          pk[e2] = pack_h2(p0 * vn_s[j0], p1 * vn_s[j0 + 1]);
        }
        *reinterpret_cast<uint4*>(p_b + swz<M>(r, 32 * kh + 8 * c8)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
      }
      l += (ls[0] + ls[1]) + (ls[2] + ls[3]);
      warp_arrive_smem(p_full + bp, lane);
    }
    // ---- epilogue: O / l / lambda_V, then diag(s) H (the inverse rotation); warp w's threads take
    // coordinates 64 kh .. 64 kh + 63 of their rows: a 64-point transform of their half, then the
    // last butterfly with the other half through shared memory (the V and P buffers, free now) ----
    if (ok && n_tiles > 0) {
      const bool w_ok =
          tc::mbar_wait(pv_done + (n_tiles - 1) % NB, (uint32_t)((n_tiles - 1) / NB) & 1u);
      ok = tc::bar_sync_and(pair_bar, 64, w_ok);
    }
    tc::fence_after_sync();
    if (ok && n_tiles > 0) {  // pair-uniform; the tensor-memory loads below are warp-collective
      float o[64];
#pragma unroll
      for (int c32 = 0; c32 < 2; ++c32) {
        uint32_t ov[32];
        tc::tmem_ld32(t_o + lane_base + 64 * kh + 32 * c32, ov);
#pragma unroll
        for (int e = 0; e < 32; ++e) o[32 * c32 + e] = __uint_as_float(ov[e]);
      }
#pragma unroll
      for (int len = 1; len < 64; len <<= 1) {
#pragma unroll
        for (int i = 0; i < 64; ++i) {
          if ((i & len) == 0) {
            const float x = o[i], y = o[i + len];
            o[i] = x + y;
            o[i + len] = x - y;
          }
        }
      }
      // exchange: row r's half kh at (kh, r), 16-byte chunk c at c ^ (r % 16)
      float4* xo = reinterpret_cast<float4*>(sm + Smem::vt);
#pragma unroll
      for (int c = 0; c < 16; ++c)
        xo[(kh * M + r) * 16 + (c ^ (r & 15))] = make_float4(o[4 * c], o[4 * c + 1], o[4 * c + 2], o[4 * c + 3]);
      xch[kh * M + r] = l;  // the half sums (the maxima slots are free now)
      tc::bar_sync(pair_bar, 64);
      const float lt = xch[r] + xch[M + r];
      const float inv = lt > 0.f ? a.inv_lam_v / lt : 0.f;
      const float sc = inv * inv_sqrt_dim<D>();
      // y_lo = a + b, y_hi = a - b (a, b: the transforms of coordinates 0 .. 63 and 64 .. 127)
      float* dst = a.out + ((long long)ti * Hq + kvh * G + gi) * D + 64 * kh;
#pragma unroll
      for (int c = 0; c < 16 && row_ok; ++c) {
        const float4 pt = xo[((1 - kh) * M + r) * 16 + (c ^ (r & 15))];
        const float4 mine = make_float4(o[4 * c], o[4 * c + 1], o[4 * c + 2], o[4 * c + 3]);
        // kh = 0: a = mine, b = partner; kh = 1: a = partner, b = mine
        float4 y;
        y.x = kh ? pt.x - mine.x : mine.x + pt.x;
        y.y = kh ? pt.y - mine.y : mine.y + pt.y;
        y.z = kh ? pt.z - mine.z : mine.z + pt.z;
        y.w = kh ? pt.w - mine.w : mine.w + pt.w;
        const int k0 = 64 * kh + 4 * c;
        float4 w;
        w.x = y.x * sc * (float)a.tab.signs[k0 + 0];
        w.y = y.y * sc * (float)a.tab.signs[k0 + 1];
        w.z = y.z * sc * (float)a.tab.signs[k0 + 2];
        w.w = y.w * sc * (float)a.tab.signs[k0 + 3];
        reinterpret_cast<float4*>(dst)[c] = w;
      }
    }
  }
  if (!ok && lane == 0) atomicOr(a.tab.status, kFlagTimeout);
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(tmem, kTmemCols);
}

template <int WK, int WV>
cudaError_t launch(const Args& a, int row_tiles, cudaStream_t s) {
  auto kern = prefill_kernel<WK, WV>;
  const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Smem::alloc);
  if (e != cudaSuccess) return e;
  kern<<<dim3((unsigned)row_tiles, (unsigned)a.k.H), kThreads, Smem::alloc, s>>>(a);
  return cudaGetLastError();
}

}  // namespace pf

size_t prefill_workspace(int n_tokens, int n_q_heads, int d) {
  const size_t q = (size_t)n_tokens * n_q_heads * 2 * d * 4;
  return (q + 255) / 256 * 256 + 256;  // prepared queries, then the prologue's counter words
}

cudaError_t launch_prefill(const DevTables& t, const DecodeArgs& qa, const DevView& k, const DevView& v, int layer,
                           int seq, const int32_t* block_table, int max_blocks, int start, float lam_k, float lam_v,
                           void* workspace, cudaStream_t s) {
  using namespace pf;
  const int n_tokens = qa.batch, Hq = qa.n_q_heads;
  if (n_tokens <= 0) return cudaSuccess;
  float* qprep = static_cast<float*>(workspace);
  unsigned int* counter = reinterpret_cast<unsigned int*>(static_cast<unsigned char*>(workspace) +
                                                          ((size_t)n_tokens * Hq * 2 * D * 4 + 255) / 256 * 256);
  const cudaError_t e = launch_qprep(t, qa, qprep, counter, s);
  if (e != cudaSuccess) return e;
  Args a{};
  a.k = k;
  a.v = v;
  a.tab = t;
  a.layer = layer;
  a.seq = seq;
  a.block_table = block_table;
  a.max_blocks = max_blocks;
  a.start = start;
  a.n_tokens = n_tokens;
  a.n_q_heads = Hq;
  a.G = Hq / k.H;
  a.qprep = qprep;
  a.out = qa.out;
  a.fq = wm_log2e() / lam_k;
  a.fs = wm_log2e() * kSqrtHalfPi / (float)D;
  a.inv_lam_v = 1.f / lam_v;
  const int row_tiles = (int)(((long long)n_tokens * a.G + M - 1) / M);
  switch (k.code_bits * 4 + v.code_bits) {
#define TQ_PF_CASE(WK, WV) \
  case WK * 4 + WV:        \
    return launch<WK, WV>(a, row_tiles, s);
    TQ_PF_CASE(2, 1) TQ_PF_CASE(2, 2) TQ_PF_CASE(2, 3)
    TQ_PF_CASE(3, 1) TQ_PF_CASE(3, 2) TQ_PF_CASE(3, 3)
    TQ_PF_CASE(4, 1) TQ_PF_CASE(4, 2) TQ_PF_CASE(4, 3)
#undef TQ_PF_CASE
  }
  return cudaErrorInvalidValue;
}

}  // namespace tq
