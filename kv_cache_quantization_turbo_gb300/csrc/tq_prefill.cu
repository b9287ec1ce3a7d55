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
// KV head's group), eight warps: warps 0-3 hold one row per thread.  Per tile of 64 keys:
//   1. every thread dequantises a quarter of one token: the codebook part lambda_K c[idx] and the
//      QJL sign part +-1 of K (turbo4: one table read per code byte) into two K-major operand
//      tiles [64 tokens x 128], and V^T (the
//      operand of the value product, lambda_V c_V[idx]) into [128 coordinates x 64 tokens]; the
//      per-token norms go to small arrays;
//   2. thread 0 issues the score products S_cb = (q'_hi + q'_lo) K_cb^T and
//      S_qjl = (S q'_hi + S q'_lo) K_sign^T (M 128, N 64; the query as high and low fp16 parts,
//      about 21 significant bits, with log2 e / lambda_K and log2 e sqrt(pi/2) / d folded in);
//   3. each thread reads its row of both products from tensor memory and forms
//      s_j = n_j S_cb + rnorm_j S_qjl (log2 units), masks keys after its position, keeps the
//      online softmax (running max raised lazily: the output accumulator in tensor memory is
//      rescaled only when the max passes the reference by 2^8), and writes
//      P_j = 2^(s_j - m) |v_j| as fp16 into the A operand of the value product;
//   4. thread 0 issues O += P V (M 128, N 128, K 64) into tensor memory.
// The steps of a tile follow each other (the CTA waits on each commit); the epilogue reads O,
// divides by the softmax sum and lambda_V, and applies diag(s) H (the inverse rotation) in
// registers.  Every wait on the tensor core is bounded; one that runs out sets the timeout bit.
#include <cuda_fp16.h>

#include "tq_device.cuh"
#include "tq_tc.cuh"

namespace tq {

__host__ __device__ constexpr float wm_log2e() { return 1.4426950408889634074f; }

namespace pf {

constexpr int D = 128;        // head_dim of this kernel
constexpr int M = 128;        // query rows per CTA
constexpr int NK = 64;        // keys per tile
constexpr int kThreads = 256;  // warps 0-3: one query row per thread; all 8 warps dequantise
constexpr uint32_t kTmemCols = 256;  // S_cb [0, 64), S_qjl [64, 128), O [128, 256)
constexpr float kLazy = 8.0f;  // log2 units: rescale O when the row max passes the reference by this

// Byte offset of element (row r, column k) in a K-major operand tile of R rows whose K columns
// come in 64-element (128-byte) blocks with the 128-byte swizzle: block k / 64 at 128 R bytes,
// row r at 128 r, 16-byte chunk (k % 64) / 8 at position ((k % 64) / 8) ^ (r % 8).
template <int R>
__host__ __device__ constexpr int swz(int r, int k) {
  return (k >> 6) * (128 * R) + r * 128 + ((((k >> 3) & 7) ^ (r & 7)) << 4) + (k & 7) * 2;
}
// Start offset of K step ks (16 columns) of such a tile.
template <int R>
__host__ __device__ constexpr uint32_t kstep(int ks) {
  return (uint32_t)((ks >> 2) * (128 * R) + (ks & 3) * 32);
}

struct Smem {  // byte offsets from a 1024-byte boundary
  static constexpr int q = 0;                  // q'_hi, q'_lo, (S q')_hi, (S q')_lo: [128 x 128] each
  static constexpr int kcb = 4 * M * D * 2;    // [64 x 128]
  static constexpr int ksg = kcb + NK * D * 2;  // [64 x 128]
  static constexpr int vt = ksg + NK * D * 2;   // [128 x 64]
  static constexpr int p = vt + D * NK * 2;     // [128 x 64]
  static constexpr int hdr = p + M * NK * 2;    // float kn[64], kr[64], vn[64]
  static constexpr int tab = hdr + 3 * NK * 4;  // fp16 cb_k[8], cb_v[8]
  static constexpr int kbt = tab + 32;          // turbo4 K: uint2 [256] per code byte: codebook pair, sign pair
  static constexpr int bar = kbt + 256 * 8;     // mbarriers: scores done, values done
  static constexpr int slot = bar + 16;         // tensor-memory address
  static constexpr int total = slot + 16;
  static constexpr int alloc = total + 1024;    // room to align the base
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

template <int WK, int WV>  // K code width (turbo K: index bits + 1), V code width (turbo-MSE: index bits)
__global__ void __launch_bounds__(kThreads, 1) prefill_kernel(const __grid_constant__ Args a) {
  constexpr int BK = WK - 1;  // K index bits; bit BK of a K code is the QJL sign
  extern __shared__ __align__(16) unsigned char smem_raw[];
  unsigned char* sm = smem_raw + ((1024u - (tc::smem_addr(smem_raw) & 1023u)) & 1023u);
  const uint32_t sb = tc::smem_addr(sm);
  const int tid = threadIdx.x, warp = tid >> 5;
  float* kn_s = reinterpret_cast<float*>(sm + Smem::hdr);
  float* kr_s = kn_s + NK;
  float* vn_s = kr_s + NK;
  __half* cbk = reinterpret_cast<__half*>(sm + Smem::tab);
  __half* cbv = cbk + 8;
  uint64_t* bar_s = reinterpret_cast<uint64_t*>(sm + Smem::bar);
  uint64_t* bar_v = bar_s + 1;
  uint32_t* slot = reinterpret_cast<uint32_t*>(sm + Smem::slot);

  const int kvh = blockIdx.y, G = a.G, Hq = a.n_q_heads;
  const int row0 = blockIdx.x * M;  // first row of this CTA in the KV head's rows (token i, head g) = i G + g
  if (warp == 0) {
    tc::tmem_alloc(slot, kTmemCols);
    if (tid == 0) {
      tc::mbar_init(bar_s, 1);
      tc::mbar_init(bar_v, 1);
    }
  }
  if (tid < 8) {
    cbk[tid] = __float2half_rn(tid < (1 << BK) ? a.tab.f16_scale[BK - 1] * a.tab.centroids[(BK - 1) * 8 + tid] : 0.f);
    cbv[tid] = __float2half_rn(tid < (1 << WV) ? a.tab.f16_scale[WV - 1] * a.tab.centroids[(WV - 1) * 8 + tid] : 0.f);
  }
  if constexpr (WK == 4) {  // a byte of turbo4 K codes = two coordinates: their codebook pair and sign pair
    const float lam = a.tab.f16_scale[BK - 1];
    const float* cb = a.tab.centroids + (BK - 1) * 8;
    const uint32_t b = tid;  // 256 threads, 256 bytes
    const __half2 c2 = __floats2half2_rn(lam * cb[b & 7u], lam * cb[(b >> 4) & 7u]);
    const __half2 s2 = __floats2half2_rn((b & 8u) ? 1.f : -1.f, (b & 128u) ? 1.f : -1.f);
    *reinterpret_cast<uint2*>(sm + Smem::kbt + 8 * b) =
        make_uint2(*reinterpret_cast<const uint32_t*>(&c2), *reinterpret_cast<const uint32_t*>(&s2));
  }

  // ---- the query operands: thread = row (warps 0-3), high and low fp16 parts of q' and S q' ----
  const bool row_warp = warp < 4;
  const int r = tid & (M - 1);
  const int rho = row0 + r, ti = rho / G, gi = rho - ti * G;
  const bool row_ok = row_warp && ti < a.n_tokens;
  const int pos = a.start + ti;  // this row's position: it attends to keys 0 .. pos
  if (row_warp) {
    const float* qp = a.qprep + ((long long)ti * Hq + kvh * G + gi) * 2 * D;
#pragma unroll 1
    for (int c8 = 0; c8 < D / 8; ++c8) {
      float x[8], y[8];
      if (row_ok) {
        const float4 x0 = *reinterpret_cast<const float4*>(qp + 8 * c8), x1 = *reinterpret_cast<const float4*>(qp + 8 * c8 + 4);
        const float4 y0 = *reinterpret_cast<const float4*>(qp + D + 8 * c8),
                     y1 = *reinterpret_cast<const float4*>(qp + D + 8 * c8 + 4);
        x[0] = x0.x; x[1] = x0.y; x[2] = x0.z; x[3] = x0.w; x[4] = x1.x; x[5] = x1.y; x[6] = x1.z; x[7] = x1.w;
        y[0] = y0.x; y[1] = y0.y; y[2] = y0.z; y[3] = y0.w; y[4] = y1.x; y[5] = y1.y; y[6] = y1.z; y[7] = y1.w;
      } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) x[e] = y[e] = 0.f;
      }
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        x[e] *= a.fq;
        y[e] *= a.fs;
      }
      uint4 hx, lx, hy, ly;
      hx = make_uint4(pack_h2(x[0], x[1]), pack_h2(x[2], x[3]), pack_h2(x[4], x[5]), pack_h2(x[6], x[7]));
      lx = make_uint4(pack_h2(lo_part(x[0]), lo_part(x[1])), pack_h2(lo_part(x[2]), lo_part(x[3])),
                      pack_h2(lo_part(x[4]), lo_part(x[5])), pack_h2(lo_part(x[6]), lo_part(x[7])));
      hy = make_uint4(pack_h2(y[0], y[1]), pack_h2(y[2], y[3]), pack_h2(y[4], y[5]), pack_h2(y[6], y[7]));
      ly = make_uint4(pack_h2(lo_part(y[0]), lo_part(y[1])), pack_h2(lo_part(y[2]), lo_part(y[3])),
                      pack_h2(lo_part(y[4]), lo_part(y[5])), pack_h2(lo_part(y[6]), lo_part(y[7])));
      const int o = swz<M>(r, 8 * c8);
      *reinterpret_cast<uint4*>(sm + Smem::q + 0 * M * D * 2 + o) = hx;
      *reinterpret_cast<uint4*>(sm + Smem::q + 1 * M * D * 2 + o) = lx;
      *reinterpret_cast<uint4*>(sm + Smem::q + 2 * M * D * 2 + o) = hy;
      *reinterpret_cast<uint4*>(sm + Smem::q + 3 * M * D * 2 + o) = ly;
    }
  }
  tc::fence_async_smem();
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *slot;
  const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;  // a warp's tensor-memory lane quarter
  const uint32_t t_cb = tmem, t_q = tmem + 64, t_o = tmem + 128;

  // keys this CTA reads: up to the last row's position; keys beyond the chunk are never attended
  const int last_row = min(row0 + M, a.n_tokens * G) - 1;
  const int n_keys = a.start + last_row / G + 1;
  const int n_tiles = (n_keys + NK - 1) / NK;
  const DevView& K = a.k;
  const DevView& V = a.v;
  const long long vec_layer = (long long)K.num_pages * K.H * K.page_size;

  float m = -INFINITY, l = 0.f;
  bool ok = true;  // every bounded wait so far completed
  const int tt = tid & (NK - 1), qt = tid >> 6;  // dequantisation: token tt of the tile, coordinates 32 qt ..
  for (int jt = 0; jt < n_tiles && ok; ++jt) {
    // the previous value product has read P and V^T before they are overwritten; every wait's
    // outcome is made CTA-uniform, so that no thread leaves the loop while others wait at a barrier
    if (jt > 0) ok = tc::mbar_wait(bar_v, (uint32_t)(jt - 1) & 1u);
    ok = __syncthreads_and(ok);
    if (!ok) break;
    // ---- 1. dequantise K and V of keys 64 jt .. 64 jt + 63 ----
    {
      const int j = jt * NK + tt;
      bool valid = j < n_keys;
      long long vec = 0;
      if (valid) {
        long long page = a.seq;
        const int lp = j / K.page_size;
        if (a.block_table) {
          page = lp < a.max_blocks ? a.block_table[lp] : -1;
          if (page < 0 || page >= K.num_pages) {
            if (qt == 0) atomicOr(a.tab.status, kFlagBlockTable);
            valid = false;
          }
        }
        vec = (long long)a.layer * vec_layer + (page * K.H + kvh) * K.page_size + (j - lp * K.page_size);
      }
      constexpr int NWK = WK, NWV = WV;  // 32-bit words of this thread's 32 codes
      uint32_t wk[NWK], wv[NWV];
      if (valid) {
        const uint32_t* pk = reinterpret_cast<const uint32_t*>(K.payload + vec * K.pay_bytes) + qt * NWK;
        const uint32_t* pv = reinterpret_cast<const uint32_t*>(V.payload + vec * V.pay_bytes) + qt * NWV;
#pragma unroll
        for (int i = 0; i < NWK; ++i) wk[i] = __ldg(pk + i);
#pragma unroll
        for (int i = 0; i < NWV; ++i) wv[i] = __ldg(pv + i);
      } else {
#pragma unroll
        for (int i = 0; i < NWK; ++i) wk[i] = 0u;
#pragma unroll
        for (int i = 0; i < NWV; ++i) wv[i] = 0u;
      }
      const __half hz = __float2half_rn(0.f), hp1 = __float2half_rn(1.f), hm1 = __float2half_rn(-1.f);
#pragma unroll
      for (int c8 = 0; c8 < 4; ++c8) {  // coordinates 32 qt + 8 c8 .. + 7
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
        const int o = swz<NK>(tt, 32 * qt + 8 * c8);
        *reinterpret_cast<uint4*>(sm + Smem::kcb + o) = kcb;
        *reinterpret_cast<uint4*>(sm + Smem::ksg + o) = ksg;
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const uint32_t vc = code_at<WV, NWV>(wv, 8 * c8 + e);
          *reinterpret_cast<__half*>(sm + Smem::vt + swz<D>(32 * qt + 8 * c8 + e, tt)) = valid ? cbv[vc] : hz;
        }
      }
      if (qt == 0) {
        float n = 0.f, rn = 0.f, nv = 0.f;
        if (valid) {
          const __half* hk = reinterpret_cast<const __half*>(K.header + vec * K.hdr_bytes);
          n = __half2float(hk[0]);
          rn = __half2float(hk[1]);
          nv = __half2float(*reinterpret_cast<const __half*>(V.header + vec * V.hdr_bytes));
        }
        kn_s[tt] = valid ? n : NAN;  // NaN marks a key that is not there (masked below)
        kr_s[tt] = rn;
        vn_s[tt] = nv;
      }
    }
    tc::fence_async_smem();
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    // ---- 2. score products ----
    if (tid == 0) {
      constexpr uint32_t id64 = tc::idesc_f16_f32(M, NK);
      const uint64_t dkc = tc::desc_sw128(sb + Smem::kcb), dks = tc::desc_sw128(sb + Smem::ksg);
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks) {
        const uint64_t qa = kstep<M>(ks) >> 4, kb = kstep<NK>(ks) >> 4;
        tc::mma_f16(t_cb, tc::desc_sw128(sb + Smem::q) + qa, dkc + kb, id64, ks > 0);
        tc::mma_f16(t_cb, tc::desc_sw128(sb + Smem::q + M * D * 2) + qa, dkc + kb, id64, true);
        tc::mma_f16(t_q, tc::desc_sw128(sb + Smem::q + 2 * M * D * 2) + qa, dks + kb, id64, ks > 0);
        tc::mma_f16(t_q, tc::desc_sw128(sb + Smem::q + 3 * M * D * 2) + qa, dks + kb, id64, true);
      }
      tc::commit(bar_s);
    }
    ok = __syncthreads_and(tc::mbar_wait(bar_s, (uint32_t)jt & 1u));
    if (!ok) break;
    tc::fence_after_sync();
    // ---- 3. online softmax of this row (warps 0-3, warp-uniform); P into the value product's A operand ----
    if (row_warp) {
    float s[NK];
#pragma unroll
    for (int h2 = 0; h2 < 2; ++h2) {
      uint32_t vcb[32], vq[32];
      tc::tmem_ld32(t_cb + lane_base + 32 * h2, vcb);
      tc::tmem_ld32(t_q + lane_base + 32 * h2, vq);
#pragma unroll
      for (int e = 0; e < 32; ++e) {
        const int jj = 32 * h2 + e, j = jt * NK + jj;
        const float n = kn_s[jj];
        const float x = fmaf(n, __uint_as_float(vcb[e]), kr_s[jj] * __uint_as_float(vq[e]));
        s[jj] = (row_ok && j <= pos && !isnan(n)) ? x : -INFINITY;
      }
    }
    float mt = s[0];
#pragma unroll
    for (int jj = 1; jj < NK; ++jj) mt = fmaxf(mt, s[jj]);
    // Raise the reference when a row's max passes it by 2^kLazy.  The tensor-memory loads and
    // stores are warp-collective, so the decision is the warp's: when any row of the warp needs it,
    // every row raises its reference to its running max (a factor of 1 where that changes nothing)
    // and rescales l and its O row.
    if (__any_sync(kFull, mt > m + kLazy)) {
      const float mn = fmaxf(m, mt);
      const float al = mn == -INFINITY ? 1.f : (m == -INFINITY ? 0.f : exp2f(m - mn));
      l *= al;
      if (jt > 0) {
#pragma unroll 1
        for (int c32 = 0; c32 < D / 32; ++c32) {
          uint32_t ov[32];
          tc::tmem_ld32(t_o + lane_base + 32 * c32, ov);
#pragma unroll
          for (int e = 0; e < 32; ++e) ov[e] = __float_as_uint(__uint_as_float(ov[e]) * al);
          tc::tmem_st32(t_o + lane_base + 32 * c32, ov);
        }
        tc::tmem_wait_st();
      }
      m = mn;
    }
#pragma unroll
    for (int c8 = 0; c8 < NK / 8; ++c8) {
      uint32_t pk[4];
#pragma unroll
      for (int e2 = 0; e2 < 4; ++e2) {
        const int j0 = 8 * c8 + 2 * e2;
        const float p0 = s[j0] == -INFINITY ? 0.f : fast_ex2(s[j0] - m);
        const float p1 = s[j0 + 1] == -INFINITY ? 0.f : fast_ex2(s[j0 + 1] - m);
        l += p0 + p1;
        pk[e2] = pack_h2(p0 * vn_s[j0], p1 * vn_s[j0 + 1]);
      }
      *reinterpret_cast<uint4*>(sm + Smem::p + swz<M>(r, 8 * c8)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
    }
    }  // row warps
    tc::fence_async_smem();
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    // ---- 4. value product O += P V ----
    if (tid == 0) {
      constexpr uint32_t id128 = tc::idesc_f16_f32(M, D);
      const uint64_t dp = tc::desc_sw128(sb + Smem::p), dv = tc::desc_sw128(sb + Smem::vt);
#pragma unroll
      for (int ks = 0; ks < NK / 16; ++ks)
        tc::mma_f16(t_o, dp + (kstep<M>(ks) >> 4), dv + (kstep<D>(ks) >> 4), id128, jt > 0 || ks > 0);
      tc::commit(bar_v);
    }
  }
  if (ok && n_tiles > 0) ok = tc::mbar_wait(bar_v, (uint32_t)(n_tiles - 1) & 1u);
  ok = __syncthreads_and(ok);
  tc::fence_after_sync();
  // ---- epilogue: O / l / lambda_V, then diag(s) H (the inverse rotation), one row per thread ----
  if (ok && n_tiles > 0 && row_warp) {  // warp-uniform: the tensor-memory loads below are warp-collective
    float o[D];
#pragma unroll
    for (int c32 = 0; c32 < D / 32; ++c32) {
      uint32_t ov[32];
      tc::tmem_ld32(t_o + lane_base + 32 * c32, ov);
#pragma unroll
      for (int e = 0; e < 32; ++e) o[32 * c32 + e] = __uint_as_float(ov[e]);
    }
    const float inv = l > 0.f ? a.inv_lam_v / l : 0.f;
#pragma unroll
    for (int len = 1; len < D; len <<= 1) {
#pragma unroll
      for (int i = 0; i < D; ++i) {
        if ((i & len) == 0) {
          const float x = o[i], y = o[i + len];
          o[i] = x + y;
          o[i + len] = x - y;
        }
      }
    }
    const float sc = inv * inv_sqrt_dim<D>();
    float* dst = a.out + ((long long)ti * Hq + kvh * G + gi) * D;
#pragma unroll
    for (int c4 = 0; c4 < D / 4 && row_ok; ++c4) {
      float4 w;
      w.x = o[4 * c4 + 0] * sc * (float)a.tab.signs[4 * c4 + 0];
      w.y = o[4 * c4 + 1] * sc * (float)a.tab.signs[4 * c4 + 1];
      w.z = o[4 * c4 + 2] * sc * (float)a.tab.signs[4 * c4 + 2];
      w.w = o[4 * c4 + 3] * sc * (float)a.tab.signs[4 * c4 + 3];
      reinterpret_cast<float4*>(dst)[c4] = w;
    }
  }
  if (!ok && tid == 0) atomicOr(a.tab.status, kFlagTimeout);
  if (!ok) {  // bounded waits for what may still be in flight before the tensor memory is freed
    tc::mbar_wait(bar_s, 0u, 1 << 10);
    tc::mbar_wait(bar_v, 0u, 1 << 10);
  }
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
