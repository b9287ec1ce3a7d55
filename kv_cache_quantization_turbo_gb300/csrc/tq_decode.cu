// Decode attention over the compressed cache.
//
//   1. prologue (one CTA per query row): q' = scale * H diag(s) q  and
//      Sq' = S q'  for turbo K ("rotate q once"); q' = scale * q for q8_0 K.
//   2. split-K attention: a work item is (split of the context, KV head,
//      layer x sequence) with all G query heads of that KV head; it scores the
//      packed K against q' and Sq',
//        s_j = n_j <q', c[idx_j]> + rnorm_j sqrt(pi/2)/d <Sq', 2 sigma_j - 1>,
//      keeps an online softmax (running max m, sum l), accumulates V in the
//      rotated space as exp(s_j - m) n_j c_V[idx_j] unless that weight is below
//      skip_threshold ("TurboQuant+: 3.8x compression ...", core content item
//      4, Sparse V), and writes the partial (m, l, acc).  Up to 16 query heads
//      per KV head run on tensor cores (tq_decode_mma.cuh); a turbo-MSE format
//      used as K, or pages that are not a multiple of 16 tokens, run
//      attend_generic_kernel below.
//   3. combine (one CTA of 4 warps per query row): log-sum-exp merge of the
//      partials, acc / l, then diag(s) H back to the original space for turbo V.
#include <cmath>

#include <cuda_fp16.h>

#include "tq_device.cuh"

namespace tq {

static int next_pow2(long long v) {
  int p = 1;
  while (p < v && p < (1 << 30)) p <<= 1;
  return p;
}

DecodePlan plan_decode(int sm_count, int d, int n_layers, int batch, int n_q_heads, int max_ctx) {
  DecodePlan p{};
  // Split size: aim at ~12 work items per warp of the tensor-core kernel (counted at 16 warps
  // per SM, query heads shared by about 4 per KV head), between 256 and 4096 tokens.  Timed on
  // the 32-layer x 32K bench workload: 512-token splits beat 1024 (item count vs. load
  // balance) and 256 (per-item overhead and partial traffic).
  const long long work = (long long)max_ctx * n_layers * batch * n_q_heads;
  const long long per_item = (work + 4LL * 16 * 12 * sm_count - 1) / (4LL * 16 * 12 * sm_count);
  int st = next_pow2(per_item);
  st = st < 256 ? 256 : (st > 4096 ? 4096 : st);
  p.split_tokens = st;
  p.n_splits = max_ctx > 0 ? (max_ctx + st - 1) / st : 1;
  const long long rows = (long long)n_layers * batch * n_q_heads;
  p.qprep_floats = (size_t)rows * 2 * d;
  p.partial_floats = (size_t)rows * p.n_splits * (d + 4);
  auto al = [](size_t b) { return (b + 255) / 256 * 256; };
  p.bytes = al(p.qprep_floats * 4) + al(p.partial_floats * 4) + 256;  // + work counter
  return p;
}

namespace {

using DecodeKernelArgs = DecodeLaunch;

// ---------------------------------------------------------------------------
// 1. query prologue
// ---------------------------------------------------------------------------
// One CTA of 4 D threads per kQprepRows query rows.  Warp w < kQprepRows rotates row w (signs,
// WHT, softmax scale) into shared memory; then thread (part p, j) forms the partial sums over
// i in [p d/4, (p + 1) d/4) of (S q')_j = sum_i S_T[i][j] q'_i for every row, and the four parts
// are added in a fixed order, so each element of S is read once per CTA and used for all its rows.
// At d <= 128 all of S_T comes into shared memory by asynchronous copies requested before the
// rotation starts (its reads in flight together); at d = 256 (256 KB) the parts read it from
// global memory.  The grid lets the attention kernel that follows launch at once (programmatic
// dependent launch): that kernel builds its tables meanwhile and waits for this grid before it
// reads anything written here.
constexpr int kQprepRows = 8, kQprepParts = 4;
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
template <int D>
__host__ __device__ constexpr int qprep_smem() {
  return D <= 128 ? D * D * 4 : 0;  // S_T staged whole
}

template <int D>
__global__ void __launch_bounds__(kQprepParts * D) qprep_kernel(DecodeKernelArgs ka) {
  constexpr int E = D / 32, RQ = kQprepRows, NP = kQprepParts, T = NP * D, IP = D / NP;
  constexpr bool STAGE = qprep_smem<D>() > 0;
  static_assert(T / 32 >= RQ, "one warp per row");
  pdl_launch_dependents();
  const DecodeArgs& a = ka.a;
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const long long row0 = (long long)blockIdx.x * RQ;
  const long long rows = (long long)a.n_layers * a.batch * a.n_q_heads;
  if (blockIdx.x == 0 && threadIdx.x < 2) ka.counter[threadIdx.x] = 0u;  // work counters of the attention launches
  __shared__ __align__(16) float q_s[D][RQ];       // q'_i of the CTA's rows: row r at [i][r]
  __shared__ __align__(16) float red[NP][RQ][D];   // the parts' partial sums
  extern __shared__ __align__(16) float s_s[];     // S_T (d <= 128)
  const bool q8 = a.k.format == TQ_FMT_Q8_0;       // q8_0 K scores the unrotated q, and needs no S q
  if (STAGE && !q8) {
    const uint32_t dst = (uint32_t)__cvta_generic_to_shared(s_s);
    const char* src = reinterpret_cast<const char*>(ka.tab.S_T);
#pragma unroll
    for (int p = threadIdx.x; p < D * D / 4; p += T) cp_async16(dst + 16 * p, src + 16 * p);
    asm volatile("cp.async.commit_group;" ::: "memory");
  }
  if (w < RQ) {
    const long long row = row0 + w;
    float x[E];
#pragma unroll
    for (int e = 0; e < E; ++e) x[e] = 0.f;
    if (row < rows) {  // warp-uniform
      if (a.q_is_fp16) {
        const __half* q = static_cast<const __half*>(a.q) + io_row_of(a, row) * D;
#pragma unroll
        for (int e = 0; e < E; ++e) x[e] = __half2float(q[E * lane + e]);
      } else {
        const float* q = static_cast<const float*>(a.q) + io_row_of(a, row) * D;
#pragma unroll
        for (int e = 0; e < E; ++e) x[e] = q[E * lane + e];
      }
      if (!q8) {
#pragma unroll
        for (int e = 0; e < E; ++e) x[e] *= (float)ka.tab.signs[E * lane + e];
        warp_wht<D>(x, lane);
      }
      float* dst = ka.qprep + row * 2 * D;
#pragma unroll
      for (int e = 0; e < E; ++e) {
        x[e] *= a.softmax_scale;
        dst[E * lane + e] = x[e];
      }
    }
#pragma unroll
    for (int e = 0; e < E; ++e) q_s[E * lane + e][w] = x[e];
  }
  if (q8) return;  // block-uniform
  if (STAGE) asm volatile("cp.async.wait_group 0;" ::: "memory");
  __syncthreads();  // q_s and S_T visible to every thread
  const int j = threadIdx.x % D, part = threadIdx.x / D;
  float acc[RQ];
#pragma unroll
  for (int r = 0; r < RQ; ++r) acc[r] = 0.f;
#pragma unroll 8
  for (int k = 0; k < IP; ++k) {
    const int i = part * IP + k;
    const float sv = STAGE ? s_s[i * D + j] : __ldg(ka.tab.S_T + (size_t)i * D + j);
    const float4 qa = *reinterpret_cast<const float4*>(&q_s[i][0]);
    const float4 qb = *reinterpret_cast<const float4*>(&q_s[i][4]);
    acc[0] = fmaf(sv, qa.x, acc[0]);
    acc[1] = fmaf(sv, qa.y, acc[1]);
    acc[2] = fmaf(sv, qa.z, acc[2]);
    acc[3] = fmaf(sv, qa.w, acc[3]);
    acc[4] = fmaf(sv, qb.x, acc[4]);
    acc[5] = fmaf(sv, qb.y, acc[5]);
    acc[6] = fmaf(sv, qb.z, acc[6]);
    acc[7] = fmaf(sv, qb.w, acc[7]);
  }
#pragma unroll
  for (int r = 0; r < RQ; ++r) red[part][r][j] = acc[r];
  __syncthreads();
  // thread t < RQ D: row t / D, output j, the parts added in order
  for (int t = threadIdx.x; t < RQ * D; t += T) {
    const int r = t / D, jj = t % D;
    if (row0 + r < rows) {
      float v = red[0][r][jj];
#pragma unroll
      for (int p = 1; p < NP; ++p) v += red[p][r][jj];
      ka.qprep[(row0 + r) * 2 * D + D + jj] = v;
    }
  }
}
static_assert(kQprepRows == 8, "the S q' loop reads the rows as two float4");
inline long long qprep_blocks(long long rows) { return (rows + kQprepRows - 1) / kQprepRows; }
// The prologue over `rows` query rows (its dynamic shared memory holds the chunks of S_T).
template <int D>
cudaError_t launch_qprep_dim(const DecodeKernelArgs& ka, long long rows, cudaStream_t s) {
  constexpr int smem = qprep_smem<D>();
  if (smem > 48 * 1024) {
    const cudaError_t e = cudaFuncSetAttribute(qprep_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
  }
  qprep_kernel<D><<<(unsigned)qprep_blocks(rows), kQprepParts * D, smem, s>>>(ka);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// token addressing of the generic kernel
// ---------------------------------------------------------------------------
__device__ __forceinline__ int clamp_seq_len(const DecodeArgs& a, int b, uint32_t* status) {
  int len = a.seq_lens[b];
  if (len < 0) len = 0;
  if (len > a.max_ctx) {
    if (threadIdx.x == 0) atomicOr(status, kFlagSeqLen);
    len = a.max_ctx;
  }
  return len;
}

// Vector index of token j of sequence b (head kvh, layer) in view V, or -1.
__device__ __forceinline__ long long token_vector(const DecodeArgs& a, const DevView& V, int layer, int b, int j,
                                                  int kvh, uint32_t* status) {
  long long page;
  if (a.block_table) {
    page = a.block_table[(long long)b * a.max_blocks_per_seq + j / V.page_size];
    if (page < 0 || page >= V.num_pages) {
      atomicOr(status, kFlagBlockTable);
      return -1;
    }
  } else {
    page = b;
  }
  const long long p = j % V.page_size;
  return (((long long)layer * V.num_pages + page) * V.H + kvh) * V.page_size + p;
}

// ---------------------------------------------------------------------------
// 2. split-K attention on CUDA cores, for what the tensor-core kernel does not
//    take (a turbo-MSE format used as K, block tables over pages that are not a
//    multiple of 16 tokens): one warp per CTA;
//    lane = token while scoring, lane = coordinates while accumulating V.
// ---------------------------------------------------------------------------
constexpr int kGMax = 16;

template <int D>
__global__ void __launch_bounds__(32) attend_generic_kernel(DecodeKernelArgs ka) {
  constexpr int E = D / 32;
  const DecodeArgs& a = ka.a;
  const int lane = threadIdx.x;
  const int split = blockIdx.x, kvh = blockIdx.y;
  const int lb = blockIdx.z, layer_rel = lb / a.batch, b = lb % a.batch;
  const int layer = k_layer_of(a, layer_rel), layer_v = v_layer_of(a, layer_rel);
  const int G = ka.G;
  const int Hq = a.n_q_heads;
  // dynamic shared memory: q' [G][D], Sq' [G][D], acc [G][D], two codebooks
  extern __shared__ __align__(16) float dsm[];
  float (*qs)[D] = reinterpret_cast<float (*)[D]>(dsm);
  float (*sqs)[D] = reinterpret_cast<float (*)[D]>(dsm + ka.G * D);
  float (*acc_s)[D] = reinterpret_cast<float (*)[D]>(dsm + 2 * ka.G * D);
  float* cbk = dsm + 3 * ka.G * D;
  float* cbv = cbk + 8;

  const long long row0 = (long long)lb * Hq + (long long)kvh * G;  // first q row of this KV head
  for (int i = lane; i < G * D; i += 32) {
    const int g = i / D, k = i % D;
    qs[g][k] = ka.qprep[(row0 + g) * 2 * D + k];
    sqs[g][k] = ka.qprep[(row0 + g) * 2 * D + D + k];
    acc_s[g][k] = 0.f;
  }
  const bool k_turbo = a.k.format != TQ_FMT_Q8_0, v_turbo = a.v.format != TQ_FMT_Q8_0;
  if (lane < 8) {
    cbk[lane] = k_turbo ? ka.tab.centroids[(a.k.idx_bits - 1) * 8 + lane] : 0.f;
    cbv[lane] = v_turbo ? ka.tab.centroids[(a.v.idx_bits - 1) * 8 + lane] : 0.f;
  }
  __syncwarp();

  const int len = clamp_seq_len(a, b, ka.tab.status);
  const int t0 = split * ka.split_tokens;
  const int t1 = min(t0 + ka.split_tokens, len);
  float m[kGMax], l[kGMax];
#pragma unroll
  for (int g = 0; g < kGMax; ++g) { m[g] = -INFINITY; l[g] = 0.f; }
  const float qjl_k = kSqrtHalfPi / (float)D;
  const int kb = a.k.idx_bits, kw = a.k.code_bits, vb = a.v.idx_bits, vw = a.v.code_bits;

  for (int tb = t0; tb < t1; tb += 32) {
    const int j = tb + lane;
    const bool valid_tok = j < t1;
    float s[kGMax];
#pragma unroll
    for (int g = 0; g < kGMax; ++g) s[g] = -INFINITY;
    long long kv = valid_tok ? token_vector(a, a.k, layer, b, j, kvh, ka.tab.status) : -1;
    if (kv >= 0) {
      const unsigned char* hdr = a.k.header + kv * a.k.hdr_bytes;
      const uint32_t* w = reinterpret_cast<const uint32_t*>(a.k.payload + kv * a.k.pay_bytes);
      float am[kGMax], aq[kGMax];
#pragma unroll
      for (int g = 0; g < kGMax; ++g) { am[g] = 0.f; aq[g] = 0.f; }
      if (k_turbo) {
        for (int i = 0; i < D; ++i) {
          const uint32_t c = stream_code(w, i, kw);
          const float cv = cbk[c & ((1u << kb) - 1u)];
          const bool pos = (c >> kb) & 1u;
#pragma unroll
          for (int g = 0; g < kGMax; ++g) {
            if (g < G) {
              am[g] = fmaf(qs[g][i], cv, am[g]);
              aq[g] += pos ? sqs[g][i] : -sqs[g][i];
            }
          }
        }
        const float n = __half2float(reinterpret_cast<const __half*>(hdr)[0]);
        const float rn = a.k.has_qjl ? __half2float(reinterpret_cast<const __half*>(hdr)[1]) : 0.f;
#pragma unroll
        for (int g = 0; g < kGMax; ++g) s[g] = n * am[g] + rn * qjl_k * aq[g];
      } else {
        const int8_t* q8 = reinterpret_cast<const int8_t*>(w);
        const __half* dl = reinterpret_cast<const __half*>(hdr);
        for (int blk = 0; blk < D / 32; ++blk) {
#pragma unroll
          for (int g = 0; g < kGMax; ++g) aq[g] = 0.f;
          for (int i = 32 * blk; i < 32 * blk + 32; ++i) {
            const float qv = (float)q8[i];
#pragma unroll
            for (int g = 0; g < kGMax; ++g)
              if (g < G) aq[g] = fmaf(qs[g][i], qv, aq[g]);
          }
          const float delta = __half2float(dl[blk]);
#pragma unroll
          for (int g = 0; g < kGMax; ++g) am[g] = fmaf(delta, aq[g], am[g]);
        }
#pragma unroll
        for (int g = 0; g < kGMax; ++g) s[g] = am[g];
      }
    }
    // online softmax over this chunk of 32 tokens
    float p[kGMax];
#pragma unroll
    for (int g = 0; g < kGMax; ++g) {
      if (g < G) {
        const float cm = warp_max(s[g]);
        const float mn = fmaxf(m[g], cm);
        const float alpha = (mn == -INFINITY) ? 1.f : expf(m[g] - mn);
        p[g] = (s[g] == -INFINITY) ? 0.f : expf(s[g] - mn);
        l[g] = l[g] * alpha + warp_sum(p[g]);
        m[g] = mn;
#pragma unroll
        for (int e = 0; e < E; ++e) acc_s[g][E * lane + e] *= alpha;
      } else {
        p[g] = 0.f;
      }
    }
    // V accumulation, token by token (lane = coordinates)
    const int nt = min(32, t1 - tb);
    for (int jj = 0; jj < nt; ++jj) {
      float pj[kGMax];
      bool keep = false;
#pragma unroll
      for (int g = 0; g < kGMax; ++g) {
        pj[g] = __shfl_sync(kFull, p[g], jj);
        keep |= (g < G) && pj[g] > 0.f && pj[g] >= a.skip_threshold;
      }
      if (!keep) continue;  // warp-uniform: every V term of this token is below the threshold
      const long long vv = token_vector(a, a.v, layer_v, b, tb + jj, kvh, ka.tab.status);
      if (vv < 0) continue;
      const unsigned char* hdr = a.v.header + vv * a.v.hdr_bytes;
      const unsigned char* pay = a.v.payload + vv * a.v.pay_bytes;
      float val[E];
      if (v_turbo) {
        const float n = __half2float(reinterpret_cast<const __half*>(hdr)[0]);
#pragma unroll
        for (int e = 0; e < E; ++e)
          val[e] = n * cbv[stream_code(reinterpret_cast<const uint32_t*>(pay), E * lane + e, vw) & ((1u << vb) - 1u)];
      } else {
        const float delta = __half2float(reinterpret_cast<const __half*>(hdr)[(E * lane) / 32]);
#pragma unroll
        for (int e = 0; e < E; ++e) val[e] = (float)reinterpret_cast<const int8_t*>(pay)[E * lane + e] * delta;
      }
#pragma unroll
      for (int g = 0; g < kGMax; ++g) {
        if (g < G && pj[g] > 0.f && pj[g] >= a.skip_threshold) {
#pragma unroll
          for (int e = 0; e < E; ++e) acc_s[g][E * lane + e] = fmaf(pj[g], val[e], acc_s[g][E * lane + e]);
        }
      }
    }
  }
  // write the partial of every query head of this KV head
  for (int g = 0; g < G; ++g) {
    float* dst = ka.partial + ((row0 + g) * ka.n_splits + split) * (D + 4);
    if (lane == 0) { dst[0] = m[g]; dst[1] = l[g]; }
#pragma unroll
    for (int e = 0; e < E; ++e) dst[4 + E * lane + e] = acc_s[g][E * lane + e];
  }
}

// ---------------------------------------------------------------------------
// 3. combine
// ---------------------------------------------------------------------------
// One CTA of kCombineWarps warps per query row: warp w merges the splits w, w + kCombineWarps, ...
// in batches of CB whose loads are all in flight together, keeping its own running maximum (a batch
// rescales what came before it only when it raises that maximum); the warps' (max, sum, acc) meet
// in shared memory and warp 0 finishes the row.  Small enough (<= 64 registers) that one wave of
// CTAs covers a few thousand rows.
constexpr int kCombineWarps = 4;
template <int D>
__global__ void __launch_bounds__(32 * kCombineWarps, 8) combine_kernel(DecodeKernelArgs ka) {
  constexpr int E = D / 32, CB = D <= 128 ? 8 : 4;
  __shared__ float xs[kCombineWarps][D];
  __shared__ float ms[kCombineWarps], ls[kCombineWarps];
  pdl_wait();  // launched as a dependent of the attention grid: its partials are complete and visible
  const DecodeArgs& a = ka.a;
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const long long row = blockIdx.x;
  const long long rows = (long long)a.n_layers * a.batch * a.n_q_heads;
  if (row >= rows) return;  // block-uniform
  const int ns = ka.n_splits;
  const float* part = ka.partial + row * ns * (D + 4);
  float M = -INFINITY, L = 0.f, x[E];
#pragma unroll
  for (int e = 0; e < E; ++e) x[e] = 0.f;
  for (int s0 = w; s0 < ns; s0 += kCombineWarps * CB) {
    float mv[CB], lv[CB], xv[CB][E];
#pragma unroll
    for (int c = 0; c < CB; ++c) {
      const int sp = s0 + kCombineWarps * c;
      mv[c] = -INFINITY;  // a split past the end, or an empty one (m = -inf), weighs 0
      lv[c] = 0.f;
#pragma unroll
      for (int e = 0; e < E; ++e) xv[c][e] = 0.f;
      if (sp < ns) {
        const float* p = part + (long long)sp * (D + 4);
        mv[c] = p[0];
        lv[c] = p[1];
        if constexpr (E % 4 == 0) {  // rows of D + 4 floats: 16-byte aligned at D = 128, 256
#pragma unroll
          for (int e = 0; e < E; e += 4) {
            const float4 v = *reinterpret_cast<const float4*>(p + 4 + E * lane + e);
            xv[c][e] = v.x;
            xv[c][e + 1] = v.y;
            xv[c][e + 2] = v.z;
            xv[c][e + 3] = v.w;
          }
        } else {
#pragma unroll
          for (int e = 0; e < E; e += 2) {
            const float2 v = *reinterpret_cast<const float2*>(p + 4 + E * lane + e);
            xv[c][e] = v.x;
            xv[c][e + 1] = v.y;
          }
        }
      }
    }
    float mb = M;
#pragma unroll
    for (int c = 0; c < CB; ++c) mb = fmaxf(mb, mv[c]);
    if (mb == -INFINITY) continue;  // warp-uniform: nothing in this batch or before it
    if (mb > M) {
      const float al = M == -INFINITY ? 0.f : expf(M - mb);
      L *= al;
#pragma unroll
      for (int e = 0; e < E; ++e) x[e] *= al;
      M = mb;
    }
#pragma unroll
    for (int c = 0; c < CB; ++c) {
      const float wj = mv[c] == -INFINITY ? 0.f : expf(mv[c] - M);
      L = fmaf(lv[c], wj, L);
#pragma unroll
      for (int e = 0; e < E; ++e) x[e] = fmaf(xv[c][e], wj, x[e]);
    }
  }
  if (lane == 0) {
    ms[w] = M;
    ls[w] = L;
  }
#pragma unroll
  for (int e = 0; e < E; ++e) xs[w][E * lane + e] = x[e];
  __syncthreads();
  if (w != 0) return;
  float Mr = ms[0];
#pragma unroll
  for (int q = 1; q < kCombineWarps; ++q) Mr = fmaxf(Mr, ms[q]);
  L = 0.f;
#pragma unroll
  for (int e = 0; e < E; ++e) x[e] = 0.f;
  if (Mr != -INFINITY) {
#pragma unroll
    for (int q = 0; q < kCombineWarps; ++q) {
      if (ms[q] == -INFINITY) continue;
      const float wq = expf(ms[q] - Mr);
      L = fmaf(ls[q], wq, L);
#pragma unroll
      for (int e = 0; e < E; ++e) x[e] = fmaf(xs[q][E * lane + e], wq, x[e]);
    }
  }
  // the row's partials are dead now: drop the 128-byte lines that lie wholly inside them from L2
  // without writing them back
  {
    const uintptr_t b0 = reinterpret_cast<uintptr_t>(part), b1 = b0 + (uintptr_t)ns * (D + 4) * 4;
    for (uintptr_t ln = (b0 + 127) & ~(uintptr_t)127; ln + 128 <= b1; ln += 32 * 128) {
      const uintptr_t at = ln + 128 * lane;
      if (at + 128 <= b1) asm volatile("discard.global.L2 [%0], 128;" ::"l"(at) : "memory");
    }
  }
  const float inv = L > 0.f ? 1.f / L : 0.f;
#pragma unroll
  for (int e = 0; e < E; ++e) x[e] *= inv;
  if (a.v.format != TQ_FMT_Q8_0) {
    warp_wht<D>(x, lane);
#pragma unroll
    for (int e = 0; e < E; ++e) x[e] *= (float)ka.tab.signs[E * lane + e];
  }
  float* dst = a.out + io_row_of(a, row) * D;
#pragma unroll
  for (int e = 0; e < E; ++e) dst[E * lane + e] = x[e];
}

// K and V code widths for the tensor-core kernels (q8_0 = 0; turbo K = index bits + 1; turbo-MSE
// V = index bits), or -1 for a format they do not take.
int mma_k_width(const DevView& v) {
  if (v.format == TQ_FMT_Q8_0) return 0;
  return format_is_turbo(v.format) && v.has_qjl ? v.code_bits : -1;
}
int mma_v_width(const DevView& v) {
  if (v.format == TQ_FMT_Q8_0) return 0;
  return format_is_turbo(v.format) && !v.has_qjl ? v.code_bits : -1;
}

// The format-parameterised tensor-core kernel takes this launch: up to 16 query heads per KV head,
// pages of a multiple of 16 tokens (or a contiguous cache), an instantiated pair of code widths.
bool attend_mma_supported(const DecodeKernelArgs& ka, int d) {
  const DecodeArgs& a = ka.a;
  if (ka.G < 1 || ka.G > 16 || ka.split_tokens % 16 != 0) return false;
  if (a.block_table != nullptr && a.k.page_size % 16 != 0) return false;
  const int wk = mma_k_width(a.k), wv = mma_v_width(a.v);
  if (wk < 0 || wv < 0) return false;
  switch (d) {
    case 64: return mma_has_d64(wk, wv);
    case 128: return mma_has_d128(wk, wv);
    case 256: return mma_has_d256(wk, wv);
  }
  return false;
}

cudaError_t launch_attend_mma_heads(const DecodeKernelArgs& ka, int d, int sm_count, cudaStream_t s) {
  const int wk = mma_k_width(ka.a.k), wv = mma_v_width(ka.a.v);
  switch (d) {
    case 64: return mma_launch_d64(ka, wk, wv, sm_count, s);
    case 128: return mma_launch_d128(ka, wk, wv, sm_count, s);
    case 256: return mma_launch_d256(ka, wk, wv, sm_count, s);
  }
  return cudaErrorInvalidValue;
}

// Up to 8 query heads per KV head, or up to 16 at d <= 128: one work item per (layer x sequence,
// KV head, split), all heads scored from each dequantised tile.  9 to 16 at d = 256: each item
// runs twice, on the two halves of the KV head's query heads (ceil(G/2) and the rest),
// as consecutive values of the work counter, so the two halves of an item run at about the same
// time and the second read of each tile is served by L2: the cache is read from HBM about once.
cudaError_t launch_attend_mma(const DecodeKernelArgs& ka, int d, int sm_count, cudaStream_t s) {
  if (ka.G <= 8 || d <= 128) return launch_attend_mma_heads(ka, d, sm_count, s);  // d <= 128: 16 heads at once
  DecodeKernelArgs two = ka;
  two.g_off = 0;
  two.g_cnt = (ka.G + 1) / 2;
  two.g_halves = 2;
  return launch_attend_mma_heads(two, d, sm_count, s);
}

template <int D>
cudaError_t launch_decode_dim(const DecodeKernelArgs& ka, int sm_count, cudaStream_t s) {
  const DecodeArgs& a = ka.a;
  const long long rows = (long long)a.n_layers * a.batch * a.n_q_heads;
  const cudaError_t eq = launch_qprep_dim<D>(ka, rows, s);
  if (eq != cudaSuccess) return eq;
  if (attend_mma_supported(ka, D)) {
    const cudaError_t e = launch_attend_mma(ka, D, sm_count, s);
    if (e != cudaSuccess) return e;
    return launch_pdl(combine_kernel<D>, dim3((unsigned)rows), dim3(32 * kCombineWarps), 0, s, ka);
  }
  dim3 grid(ka.n_splits, a.k.H, a.n_layers * a.batch);
  const size_t smem = (3 * (size_t)ka.G * D + 16) * sizeof(float);
  if (smem > 48 * 1024) {
    const cudaError_t e =
        cudaFuncSetAttribute(attend_generic_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  attend_generic_kernel<D><<<grid, 32, smem, s>>>(ka);
  return launch_pdl(combine_kernel<D>, dim3((unsigned)rows), dim3(32 * kCombineWarps), 0, s, ka);
}

}  // namespace

cudaError_t launch_qprep(const DevTables& t, const DecodeArgs& a, float* qprep, unsigned int* counter,
                         cudaStream_t s) {
  DecodeKernelArgs ka{};
  ka.a = a;
  ka.tab = t;
  ka.qprep = qprep;
  ka.counter = counter;
  const long long rows = (long long)a.n_layers * a.batch * a.n_q_heads;
  if (rows <= 0) return cudaSuccess;
  switch (t.d) {
    case 64: return launch_qprep_dim<64>(ka, rows, s);
    case 128: return launch_qprep_dim<128>(ka, rows, s);
    case 256: return launch_qprep_dim<256>(ka, rows, s);
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

cudaError_t launch_decode(const DevTables& t, const DecodeArgs& a, const DecodePlan& plan, void* workspace,
                          int sm_count, cudaStream_t s) {
  DecodeKernelArgs ka;
  ka.a = a;
  ka.tab = t;
  ka.split_tokens = plan.split_tokens;
  ka.n_splits = plan.n_splits;
  ka.G = a.n_q_heads / a.k.H;
  ka.g_off = 0;
  ka.g_cnt = ka.G;
  ka.g_halves = 1;
  unsigned char* ws = static_cast<unsigned char*>(workspace);
  ka.qprep = reinterpret_cast<float*>(ws);
  ka.partial = reinterpret_cast<float*>(ws + (plan.qprep_floats * 4 + 255) / 256 * 256);
  ka.counter = reinterpret_cast<unsigned int*>(ws + (plan.qprep_floats * 4 + 255) / 256 * 256 +
                                               (plan.partial_floats * 4 + 255) / 256 * 256);
  ka.keep_partials = plan.partial_floats * 4 <= kKeepPartialsMaxBytes ? 1 : 0;
  switch (t.d) {
    case 64: return launch_decode_dim<64>(ka, sm_count, s);
    case 128: return launch_decode_dim<128>(ka, sm_count, s);
    case 256: return launch_decode_dim<256>(ka, sm_count, s);
  }
  return cudaErrorInvalidValue;
}

}  // namespace tq
