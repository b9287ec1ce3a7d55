// Host side of libtq: sizes, the Lloyd-Max codebook, the default random
// tables, contexts, argument validation and the exported C entry points.
// Every device step runs in the kernels of tq_encode.cu / tq_decode.cu /
// tq_dequant.cu; nothing here computes on the data path.
#include <cmath>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <new>
#include <algorithm>
#include <vector>

#include <cuda_fp16.h>

#include "tq_internal.h"

using namespace tq;

// ---------------------------------------------------------------------------
// formats and sizes
// ---------------------------------------------------------------------------

namespace tq {

bool format_is_turbo(int f) { return f >= TQ_FMT_TURBO2 && f <= TQ_FMT_TURBO4_MSE; }
bool format_has_qjl(int f) { return f >= TQ_FMT_TURBO2 && f <= TQ_FMT_TURBO4; }

// Stage-1 index bits of a turbo format ("TurboQuant+ KV cache compression",
// format table: turbo2/3/4 = 1/2/3 bits + 1 QJL bit; the _MSE forms drop the
// QJL bit), the min-max bit width, or 8 for q8_0.
int format_idx_bits(int f, int minmax_bits) {
  switch (f) {
    case TQ_FMT_TURBO2: case TQ_FMT_TURBO2_MSE: return 1;
    case TQ_FMT_TURBO3: case TQ_FMT_TURBO3_MSE: return 2;
    case TQ_FMT_TURBO4: case TQ_FMT_TURBO4_MSE: return 3;
    case TQ_FMT_Q8_0: return 8;
    case TQ_FMT_MINMAX: return (minmax_bits >= 2 && minmax_bits <= 4) ? minmax_bits : 0;
    default: return 0;
  }
}

static bool dim_ok(int d) { return d == 64 || d == 128 || d == 256; }

bool make_dev_view(const tq_cache_view* v, DevView* o) {
  if (!v || !o) return false;
  const int f = v->format;
  const int b = format_idx_bits(f, v->bits);
  if (b == 0 || !dim_ok(v->head_dim) || v->n_kv_heads < 1 || v->page_size < 1 || v->num_pages < 1 ||
      v->n_layers < 1 || !v->payload || !v->header)
    return false;
  if ((reinterpret_cast<uintptr_t>(v->payload) & 15) || (reinterpret_cast<uintptr_t>(v->header) & 3))
    return false;
  o->format = f;
  o->d = v->head_dim;
  o->H = v->n_kv_heads;
  o->page_size = v->page_size;
  o->num_pages = v->num_pages;
  o->n_layers = v->n_layers;
  o->idx_bits = b;
  o->has_qjl = format_has_qjl(f) ? 1 : 0;
  o->code_bits = format_is_turbo(f) ? b + o->has_qjl : b;
  o->pay_bytes = (int)tq_payload_bytes((tq_format)f, v->head_dim, v->bits);
  o->hdr_bytes = (int)tq_header_bytes((tq_format)f, v->head_dim, v->bits);
  o->payload = static_cast<unsigned char*>(v->payload);
  o->header = static_cast<unsigned char*>(v->header);
  return o->pay_bytes > 0 && o->hdr_bytes > 0;
}

}  // namespace tq

extern "C" {

const char* tq_status_string(tq_status s) {
  switch (s) {
    case TQ_OK: return "ok";
    case TQ_ERR_INVALID_ARG: return "invalid argument";
    case TQ_ERR_UNSUPPORTED: return "unsupported";
    case TQ_ERR_WORKSPACE: return "workspace too small";
    case TQ_ERR_CUDA: return "CUDA error";
    case TQ_ERR_OOM: return "out of memory";
  }
  return "unknown status";
}

const char* tq_format_name(tq_format f) {
  switch (f) {
    case TQ_FMT_TURBO2: return "turbo2";
    case TQ_FMT_TURBO3: return "turbo3";
    case TQ_FMT_TURBO4: return "turbo4";
    case TQ_FMT_TURBO2_MSE: return "turbo2_mse";
    case TQ_FMT_TURBO3_MSE: return "turbo3_mse";
    case TQ_FMT_TURBO4_MSE: return "turbo4_mse";
    case TQ_FMT_Q8_0: return "q8_0";
    case TQ_FMT_MINMAX: return "minmax";
  }
  return "unknown";
}

size_t tq_payload_bytes(tq_format f, int head_dim, int bits) {
  const int b = format_idx_bits(f, bits);
  if (b == 0 || head_dim < 64 || (head_dim & (head_dim - 1)) || head_dim > kMaxDim) return 0;
  if (f == TQ_FMT_Q8_0) return (size_t)head_dim;
  const int w = format_is_turbo(f) ? b + (format_has_qjl(f) ? 1 : 0) : b;
  return (size_t)head_dim * w / 8;
}

size_t tq_header_bytes(tq_format f, int head_dim, int bits) {
  if (tq_payload_bytes(f, head_dim, bits) == 0) return 0;
  if (f == TQ_FMT_Q8_0) return (size_t)head_dim / 32 * 2;
  if (f == TQ_FMT_MINMAX) return (size_t)head_dim / 64 * 4;
  return format_has_qjl(f) ? 4 : 2;
}

size_t tq_vector_bytes(tq_format f, int head_dim, int bits) {
  return tq_payload_bytes(f, head_dim, bits) + tq_header_bytes(f, head_dim, bits);
}

// ---------------------------------------------------------------------------
// Lloyd-Max codebook for N(0, 1/d)
// ---------------------------------------------------------------------------

static double npdf(double t) { return std::exp(-0.5 * t * t) * 0.39894228040143267794; }
static double ncdf(double t) { return 0.5 * std::erfc(-t * 0.70710678118654752440); }

// inverse of ncdf by bisection (start values only)
static double ninv(double p) {
  double lo = -40.0, hi = 40.0;
  for (int i = 0; i < 200; ++i) {
    const double mid = 0.5 * (lo + hi);
    (ncdf(mid) < p ? lo : hi) = mid;
  }
  return 0.5 * (lo + hi);
}

tq_status tq_codebook_build(int bits, int head_dim, float* centroids, float* boundaries) {
  if (bits < 1 || bits > 4 || head_dim < 1 || !centroids || (!boundaries && bits > 0)) return TQ_ERR_INVALID_ARG;
  const int L = 1 << bits;
  double c[16], b[16];
  for (int k = 0; k < L; ++k) c[k] = ninv((k + 0.5) / L);
  // Lloyd iteration in units of sigma: cells [b_{k-1}, b_k), centroid = E[X | cell]
  for (int it = 0; it < 200000; ++it) {
    for (int k = 0; k + 1 < L; ++k) b[k] = 0.5 * (c[k] + c[k + 1]);
    double moved = 0.0;
    for (int k = 0; k < L; ++k) {
      const double lo = (k == 0) ? -INFINITY : b[k - 1];
      const double hi = (k == L - 1) ? INFINITY : b[k];
      const double plo = std::isinf(lo) ? 0.0 : npdf(lo), phi_ = std::isinf(hi) ? 0.0 : npdf(hi);
      const double mass = (std::isinf(hi) ? 1.0 : ncdf(hi)) - (std::isinf(lo) ? 0.0 : ncdf(lo));
      const double cn = (plo - phi_) / mass;
      moved = std::fmax(moved, std::fabs(cn - c[k]));
      c[k] = cn;
    }
    if (moved < 1e-13) break;
  }
  // The density is symmetric, so the optimal quantiser is odd: mirror the two
  // halves so that rounding cannot shift the middle boundary off zero.
  for (int k = 0; k < L / 2; ++k) {
    const double a = 0.5 * (c[L - 1 - k] - c[k]);
    c[k] = -a;
    c[L - 1 - k] = a;
  }
  const double sigma = 1.0 / std::sqrt((double)head_dim);
  for (int k = 0; k < L; ++k) centroids[k] = (float)(c[k] * sigma);
  for (int k = 0; k + 1 < L; ++k) boundaries[k] = (float)(0.5 * (c[k] + c[k + 1]) * sigma);
  return TQ_OK;
}

// Scale lambda in [1, 2) that makes every lambda * |centroid| (an fp32 product)
// round to fp16 with the smallest worst relative error.  The tensor-core decode
// kernel keeps codebook values in fp16 tables; plain rounding errs by up to
// 2^-11 relative, the same for every token with the same index, so it does not
// average out.  With lambda chosen over 2^20 candidates the worst error is
// ~1e-5; the kernel divides lambda back out of the per-token norm.
static float best_f16_scale(const float* c, int L) {
  float best = 1.0f;
  double best_err = 1e30;
  for (int i = 0; i < (1 << 20); ++i) {
    const float lam = 1.0f + (float)i * 0x1.0p-20f;
    double worst = 0.0;
    for (int k = L / 2; k < L; ++k) {
      const float p = lam * c[k];
      const float h = __half2float(__float2half_rn(p));
      worst = std::fmax(worst, std::fabs((double)h - (double)p) / std::fabs((double)p));
      if (worst >= best_err) break;
    }
    if (worst < best_err) {
      best_err = worst;
      best = lam;
    }
  }
  return best;
}

// ---------------------------------------------------------------------------
// default random tables (SplitMix64, counter based)
// ---------------------------------------------------------------------------

static uint64_t splitmix64_at(uint64_t c) {
  uint64_t z = c + 0x9E3779B97F4A7C15ull;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

tq_status tq_signs_generate(uint32_t seed, int head_dim, int8_t* signs) {
  if (head_dim < 1 || !signs) return TQ_ERR_INVALID_ARG;
  const uint64_t base = (uint64_t)seed << 32;
  for (int i = 0; i < head_dim; ++i) signs[i] = (splitmix64_at(base + (uint64_t)i) >> 63) ? -1 : 1;
  return TQ_OK;
}

tq_status tq_qjl_matrix_generate(uint32_t seed, int head_dim, float* S) {
  if (head_dim < 1 || head_dim > kMaxDim || !S) return TQ_ERR_INVALID_ARG;
  const uint64_t base = (uint64_t)seed << 32;
  const double two_pi = 6.283185307179586476925;
  for (uint64_t e = 0; e < (uint64_t)head_dim * head_dim; ++e) {
    const double u1 = ((double)(splitmix64_at(base + 2 * e) >> 11) + 1.0) * 0x1.0p-53;
    const double u2 = ((double)(splitmix64_at(base + 2 * e + 1) >> 11) + 1.0) * 0x1.0p-53;
    S[e] = (float)(std::sqrt(-2.0 * std::log(u1)) * std::cos(two_pi * u2));
  }
  return TQ_OK;
}

// ---------------------------------------------------------------------------
// context
// ---------------------------------------------------------------------------

tq_status tq_context_create(int head_dim, uint32_t wht_seed, uint32_t qjl_seed, const int8_t* signs,
                            const float* qjl, tq_context** out) {
  if (!out) return TQ_ERR_INVALID_ARG;
  *out = nullptr;
  if (head_dim != 64 && head_dim != 128 && head_dim != 256) return TQ_ERR_UNSUPPORTED;
  if (signs)
    for (int i = 0; i < head_dim; ++i)
      if (signs[i] != 1 && signs[i] != -1) return TQ_ERR_INVALID_ARG;
  tq_context* ctx = new (std::nothrow) tq_context();
  if (!ctx) return TQ_ERR_OOM;
  const int d = head_dim;
  ctx->d = d;
  ctx->wht_seed = wht_seed;
  ctx->qjl_seed = qjl_seed;
  if (cudaGetDevice(&ctx->device) != cudaSuccess ||
      cudaDeviceGetAttribute(&ctx->sm_count, cudaDevAttrMultiProcessorCount, ctx->device) != cudaSuccess) {
    delete ctx;
    return TQ_ERR_CUDA;
  }
  ctx->S_h = static_cast<float*>(std::malloc(sizeof(float) * d * d));
  if (!ctx->S_h) { delete ctx; return TQ_ERR_OOM; }
  if (signs) std::memcpy(ctx->signs_h, signs, d);
  else tq_signs_generate(wht_seed, d, ctx->signs_h);
  if (qjl) std::memcpy(ctx->S_h, qjl, sizeof(float) * d * d);
  else tq_qjl_matrix_generate(qjl_seed, d, ctx->S_h);
  std::memset(ctx->centroids_h, 0, sizeof(ctx->centroids_h));
  std::memset(ctx->boundaries_h, 0, sizeof(ctx->boundaries_h));
  for (int b = 1; b <= 3; ++b) {
    tq_codebook_build(b, d, ctx->centroids_h[b - 1], ctx->boundaries_h[b - 1]);
    ctx->f16_scale_h[b - 1] = best_f16_scale(ctx->centroids_h[b - 1], 1 << b);
  }

  // one device block: status | signs | centroids | boundaries | f16 scales | S | S_T | S fragments
  const size_t off_signs = 256, off_cent = off_signs + 256, off_bnd = off_cent + 256,
               off_scale = off_bnd + 256, off_S = off_scale + 256, off_ST = off_S + sizeof(float) * d * d,
               off_SF = off_ST + sizeof(float) * d * d, total = off_SF + sizeof(uint32_t) * d * d;
  std::vector<unsigned char> host(total, 0);
  std::memcpy(host.data() + off_signs, ctx->signs_h, d);
  std::memcpy(host.data() + off_cent, ctx->centroids_h, sizeof(ctx->centroids_h));
  std::memcpy(host.data() + off_bnd, ctx->boundaries_h, sizeof(ctx->boundaries_h));
  std::memcpy(host.data() + off_scale, ctx->f16_scale_h, sizeof(ctx->f16_scale_h));
  std::memcpy(host.data() + off_S, ctx->S_h, sizeof(float) * d * d);
  float* st = reinterpret_cast<float*>(host.data() + off_ST);
  for (int j = 0; j < d; ++j)
    for (int i = 0; i < d; ++i) st[i * d + j] = ctx->S_h[j * d + i];
  {
    // hi/lo fp16 split of S in B-fragment order (tensor-core projection of the encoder)
    uint32_t* sf = reinterpret_cast<uint32_t*>(host.data() + off_SF);
    auto pair = [&](int row, int col, bool lo) -> uint32_t {
      uint32_t r = 0;
      for (int k = 0; k < 2; ++k) {
        const float v = ctx->S_h[row * d + col + k];
        const __half h = __float2half_rn(v);
        const __half x = lo ? __float2half_rn(v - __half2float(h)) : h;
        r |= (uint32_t)__half_as_ushort(x) << (16 * k);
      }
      return r;
    };
    for (int nb = 0; nb < d / 8; ++nb)
      for (int ks = 0; ks < d / 16; ++ks)
        for (int lane = 0; lane < 32; ++lane) {
          const int row = 8 * nb + lane / 4, col = 16 * ks + 2 * (lane % 4);
          uint32_t* e = sf + 4 * ((size_t)(nb * (d / 16) + ks) * 32 + lane);
          e[0] = pair(row, col, false);
          e[1] = pair(row, col + 8, false);
          e[2] = pair(row, col, true);
          e[3] = pair(row, col + 8, true);
        }
  }
  if (cudaMalloc(&ctx->dev_block, total) != cudaSuccess) {
    std::free(ctx->S_h);
    delete ctx;
    return TQ_ERR_OOM;
  }
  if (cudaMemcpy(ctx->dev_block, host.data(), total, cudaMemcpyHostToDevice) != cudaSuccess) {
    cudaFree(ctx->dev_block);
    std::free(ctx->S_h);
    delete ctx;
    return TQ_ERR_CUDA;
  }
  unsigned char* base = static_cast<unsigned char*>(ctx->dev_block);
  ctx->tables.d = d;
  ctx->tables.status = reinterpret_cast<uint32_t*>(base);
  ctx->tables.signs = reinterpret_cast<const int8_t*>(base + off_signs);
  ctx->tables.centroids = reinterpret_cast<const float*>(base + off_cent);
  ctx->tables.boundaries = reinterpret_cast<const float*>(base + off_bnd);
  ctx->tables.f16_scale = reinterpret_cast<const float*>(base + off_scale);
  ctx->tables.S = reinterpret_cast<const float*>(base + off_S);
  ctx->tables.S_T = reinterpret_cast<const float*>(base + off_ST);
  ctx->tables.S_frag = reinterpret_cast<const uint4*>(base + off_SF);
  *out = ctx;
  return TQ_OK;
}

tq_status tq_context_destroy(tq_context* ctx) {
  if (!ctx) return TQ_ERR_INVALID_ARG;
  int cur = -1;
  cudaGetDevice(&cur);
  if (cur != ctx->device) cudaSetDevice(ctx->device);
  const cudaError_t e = cudaFree(ctx->dev_block);
  if (cur >= 0 && cur != ctx->device) cudaSetDevice(cur);
  std::free(ctx->S_h);
  delete ctx;
  return e == cudaSuccess ? TQ_OK : TQ_ERR_CUDA;
}

tq_status tq_context_get_tables(const tq_context* ctx, int8_t* signs, float* qjl, float* centroids,
                                float* boundaries) {
  if (!ctx) return TQ_ERR_INVALID_ARG;
  if (signs) std::memcpy(signs, ctx->signs_h, ctx->d);
  if (qjl) std::memcpy(qjl, ctx->S_h, sizeof(float) * ctx->d * ctx->d);
  if (centroids) std::memcpy(centroids, ctx->centroids_h, sizeof(ctx->centroids_h));
  if (boundaries) std::memcpy(boundaries, ctx->boundaries_h, sizeof(ctx->boundaries_h));
  return TQ_OK;
}

tq_status tq_get_status(tq_context* ctx, uint32_t* flags) {
  if (!ctx) return TQ_ERR_INVALID_ARG;
  uint32_t v = 0;
  if (cudaMemcpy(&v, ctx->tables.status, 4, cudaMemcpyDeviceToHost) != cudaSuccess) return TQ_ERR_CUDA;
  if (v && cudaMemset(ctx->tables.status, 0, 4) != cudaSuccess) return TQ_ERR_CUDA;
  if (flags) *flags = v;
  return v ? TQ_ERR_INVALID_ARG : TQ_OK;
}

// ---------------------------------------------------------------------------
// encode / dequantize / decode entry points
// ---------------------------------------------------------------------------

static tq_status cuda_status(cudaError_t e) { return e == cudaSuccess ? TQ_OK : TQ_ERR_CUDA; }

tq_status tq_encode_kv(const tq_context* ctx, const tq_cache_view* k_view, const void* k,
                       const tq_cache_view* v_view, const void* v, int layer_begin, int n_layers,
                       int n_tokens, int64_t in_layer_stride, int64_t in_token_stride,
                       const int64_t* slots, int64_t slot_begin, tq_stream_t stream) {
  if (!ctx || (!k_view && !v_view)) return TQ_ERR_INVALID_ARG;
  if (n_layers < 0 || n_tokens < 0 || layer_begin < 0 || slot_begin < 0) return TQ_ERR_INVALID_ARG;
  DevView kv{}, vv{};
  const int d = ctx->d;
  if (k_view) {
    if (!k || !make_dev_view(k_view, &kv)) return TQ_ERR_INVALID_ARG;
    if (kv.d != d) return TQ_ERR_INVALID_ARG;
    if (format_is_turbo(kv.format) && !kv.has_qjl) return TQ_ERR_INVALID_ARG;  // K needs the QJL stage
    if (layer_begin + n_layers > kv.n_layers) return TQ_ERR_INVALID_ARG;
  }
  if (v_view) {
    if (!v || !make_dev_view(v_view, &vv)) return TQ_ERR_INVALID_ARG;
    if (vv.d != d) return TQ_ERR_INVALID_ARG;
    if (layer_begin + n_layers > vv.n_layers) return TQ_ERR_INVALID_ARG;
  }
  if (k_view && v_view && kv.H != vv.H) return TQ_ERR_INVALID_ARG;
  const int H = k_view ? kv.H : vv.H;
  if (in_token_stride < (int64_t)H * d || (n_layers > 1 && in_layer_stride < in_token_stride * n_tokens))
    return TQ_ERR_INVALID_ARG;
  // the kernels read inputs with 16-byte vector loads
  if ((reinterpret_cast<uintptr_t>(k) & 15) || (reinterpret_cast<uintptr_t>(v) & 15) || (in_token_stride & 7) ||
      (n_layers > 1 && (in_layer_stride & 7)))
    return TQ_ERR_INVALID_ARG;
  if (n_layers == 0 || n_tokens == 0) return TQ_OK;
  if ((int64_t)n_layers * n_tokens * H >= (int64_t(1) << 32)) return TQ_ERR_UNSUPPORTED;  // split the call
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (k_view) {
    const cudaError_t e = launch_encode(ctx->tables, kv, static_cast<const __half*>(k), layer_begin, n_layers,
                                        n_tokens, in_layer_stride, in_token_stride,
                                        reinterpret_cast<const long long*>(slots), slot_begin, ctx->sm_count, s);
    if (e != cudaSuccess) return TQ_ERR_CUDA;
  }
  if (v_view) {
    const cudaError_t e = launch_encode(ctx->tables, vv, static_cast<const __half*>(v), layer_begin, n_layers,
                                        n_tokens, in_layer_stride, in_token_stride,
                                        reinterpret_cast<const long long*>(slots), slot_begin, ctx->sm_count, s);
    if (e != cudaSuccess) return TQ_ERR_CUDA;
  }
  return TQ_OK;
}

tq_status tq_dequantize(const tq_context* ctx, const tq_cache_view* view, int layer, const int64_t* slots,
                        int64_t slot_begin, int n, int include_qjl, float* out, tq_stream_t stream) {
  DevView dv{};
  if (!ctx || !out || n < 0 || slot_begin < 0 || !make_dev_view(view, &dv)) return TQ_ERR_INVALID_ARG;
  if (dv.d != ctx->d || layer < 0 || layer >= dv.n_layers) return TQ_ERR_INVALID_ARG;
  if (n == 0) return TQ_OK;
  return cuda_status(launch_dequant(ctx->tables, dv, layer, reinterpret_cast<const long long*>(slots), slot_begin,
                                    n, include_qjl, out, reinterpret_cast<cudaStream_t>(stream)));
}

size_t tq_decode_workspace_bytes(const tq_context* ctx, int n_layers, int batch, int n_q_heads, int max_ctx) {
  if (!ctx || n_layers < 1 || batch < 1 || n_q_heads < 1 || max_ctx < 0) return 0;
  return plan_decode(ctx->sm_count, ctx->d, n_layers, batch, n_q_heads, max_ctx).bytes;
}

tq_status tq_decode_attention(const tq_context* ctx, const void* q, int q_is_fp16, int n_layers, int batch,
                              int n_q_heads, const tq_cache_view* k_view, const tq_cache_view* v_view,
                              int layer_begin, const int32_t* seq_lens, int max_ctx, const int32_t* block_table,
                              int max_blocks_per_seq, float softmax_scale, float skip_threshold,
                              void* workspace, size_t workspace_bytes, float* out, tq_stream_t stream) {
  if (!ctx || !q || !out || !seq_lens || !k_view || !v_view) return TQ_ERR_INVALID_ARG;
  if (n_layers < 0 || batch < 0 || n_q_heads < 1 || layer_begin < 0 || max_ctx < 0) return TQ_ERR_INVALID_ARG;
  if (q_is_fp16 != 0 && q_is_fp16 != 1) return TQ_ERR_INVALID_ARG;
  if (!std::isfinite(softmax_scale) || !(skip_threshold >= 0.0f) || !std::isfinite(skip_threshold))
    return TQ_ERR_INVALID_ARG;
  DecodeArgs a{};
  if (!make_dev_view(k_view, &a.k) || !make_dev_view(v_view, &a.v)) return TQ_ERR_INVALID_ARG;
  const int d = ctx->d;
  if (a.k.d != d || a.v.d != d || a.k.H != a.v.H) return TQ_ERR_INVALID_ARG;
  if (a.k.page_size != a.v.page_size || a.k.num_pages != a.v.num_pages) return TQ_ERR_INVALID_ARG;
  if (layer_begin + n_layers > a.k.n_layers || layer_begin + n_layers > a.v.n_layers) return TQ_ERR_INVALID_ARG;
  if (n_q_heads % a.k.H != 0 || n_q_heads / a.k.H > 16) return TQ_ERR_UNSUPPORTED;
  const bool k_ok = format_is_turbo(a.k.format) || a.k.format == TQ_FMT_Q8_0;
  const bool v_ok = (format_is_turbo(a.v.format) && !a.v.has_qjl) || a.v.format == TQ_FMT_Q8_0;
  if (!k_ok || !v_ok) return TQ_ERR_UNSUPPORTED;
  if (block_table) {
    if (max_blocks_per_seq < 1 || (int64_t)max_blocks_per_seq * a.k.page_size < max_ctx) return TQ_ERR_INVALID_ARG;
  } else if (max_ctx > a.k.page_size || batch > a.k.num_pages) {
    return TQ_ERR_INVALID_ARG;  // contiguous: sequence b is page b of capacity page_size
  }
  if (n_layers == 0 || batch == 0) return TQ_OK;
  const DecodePlan plan = plan_decode(ctx->sm_count, d, n_layers, batch, n_q_heads, max_ctx);
  if (!workspace || workspace_bytes < plan.bytes || (reinterpret_cast<uintptr_t>(workspace) & 255))
    return TQ_ERR_WORKSPACE;
  a.q = q;
  a.q_is_fp16 = q_is_fp16;
  a.n_layers = n_layers;
  a.batch = batch;
  a.n_q_heads = n_q_heads;
  a.layer_begin = layer_begin;
  a.seq_lens = seq_lens;
  a.max_ctx = max_ctx;
  a.block_table = block_table;
  a.max_blocks_per_seq = block_table ? max_blocks_per_seq : 1;
  a.softmax_scale = softmax_scale;
  a.skip_threshold = skip_threshold;
  a.out = out;
  return cuda_status(launch_decode(ctx->tables, a, plan, workspace, ctx->sm_count,
                                   reinterpret_cast<cudaStream_t>(stream)));
}

// ---------------------------------------------------------------------------
// per-layer views (a format per layer, e.g. Boundary V)
// ---------------------------------------------------------------------------

// The view of one layer: the view with its arrays advanced to layer `layer` and n_layers = 1.
static bool layer_view(const tq_cache_view* v, int layer, int run, DevView* out) {
  if (!make_dev_view(v, out) || layer < 0 || run < 1 || layer + run > out->n_layers) return false;
  const long long vecs = (long long)out->num_pages * out->H * out->page_size;
  out->payload += (size_t)layer * vecs * out->pay_bytes;
  out->header += (size_t)layer * vecs * out->hdr_bytes;
  out->n_layers = run;
  return true;
}

static bool same_view(const tq_cache_view& a, const tq_cache_view& b) {
  return a.format == b.format && a.head_dim == b.head_dim && a.n_kv_heads == b.n_kv_heads &&
         a.page_size == b.page_size && a.num_pages == b.num_pages && a.n_layers == b.n_layers && a.bits == b.bits &&
         a.payload == b.payload && a.header == b.header;
}

// Length of the run of layers from l that share their views at consecutive view layers.
static int layer_run(const tq_cache_view* kv, const int32_t* kl, const tq_cache_view* vv, const int32_t* vl, int l,
                     int n) {
  int r = l + 1;
  while (r < n && (!kv || (same_view(kv[r], kv[l]) && kl[r] == kl[r - 1] + 1)) &&
         (!vv || (same_view(vv[r], vv[l]) && vl[r] == vl[r - 1] + 1)))
    ++r;
  return r - l;
}

tq_status tq_encode_kv_layers(const tq_context* ctx, const tq_cache_view* k_views, const int32_t* k_view_layers,
                              const tq_cache_view* v_views, const int32_t* v_view_layers, int n_layers,
                              const void* k, const void* v, int n_tokens, int64_t in_layer_stride,
                              int64_t in_token_stride, const int64_t* slots, int64_t slot_begin, tq_stream_t stream) {
  if (!ctx || n_layers < 0 || (!k_views && !v_views)) return TQ_ERR_INVALID_ARG;
  if ((k_views && (!k_view_layers || !k)) || (v_views && (!v_view_layers || !v))) return TQ_ERR_INVALID_ARG;
  // every layer validated before anything is launched
  for (int l = 0; l < n_layers; ++l) {
    DevView dv{};
    if (k_views && !layer_view(&k_views[l], k_view_layers[l], 1, &dv)) return TQ_ERR_INVALID_ARG;
    if (v_views && !layer_view(&v_views[l], v_view_layers[l], 1, &dv)) return TQ_ERR_INVALID_ARG;
  }
  const size_t esz = 2;  // fp16 inputs
  for (int l = 0; l < n_layers;) {
    const int run = layer_run(k_views, k_view_layers, v_views, v_view_layers, l, n_layers);
    const unsigned char* kp = static_cast<const unsigned char*>(k);
    const unsigned char* vp = static_cast<const unsigned char*>(v);
    // one call of tq_encode_kv per run: K and V of the run may sit at different layers of their views,
    // so they go as two calls when they do
    const int kb = k_views ? k_view_layers[l] : 0, vb = v_views ? v_view_layers[l] : 0;
    tq_status st = TQ_OK;
    if (k_views && v_views && kb == vb) {
      st = tq_encode_kv(ctx, &k_views[l], kp + (size_t)l * in_layer_stride * esz, &v_views[l],
                        vp + (size_t)l * in_layer_stride * esz, kb, run, n_tokens, in_layer_stride, in_token_stride,
                        slots, slot_begin, stream);
    } else {
      if (k_views)
        st = tq_encode_kv(ctx, &k_views[l], kp + (size_t)l * in_layer_stride * esz, nullptr, nullptr, kb, run,
                          n_tokens, in_layer_stride, in_token_stride, slots, slot_begin, stream);
      if (st == TQ_OK && v_views)
        st = tq_encode_kv(ctx, nullptr, nullptr, &v_views[l], vp + (size_t)l * in_layer_stride * esz, vb, run,
                          n_tokens, in_layer_stride, in_token_stride, slots, slot_begin, stream);
    }
    if (st != TQ_OK) return st;
    l += run;
  }
  return TQ_OK;
}

tq_status tq_decode_attention_layers(const tq_context* ctx, const void* q, int q_is_fp16, int n_layers, int batch,
                                     int n_q_heads, const tq_cache_view* k_views, const int32_t* k_view_layers,
                                     const tq_cache_view* v_views, const int32_t* v_view_layers,
                                     const int32_t* seq_lens, int max_ctx, const int32_t* block_table,
                                     int max_blocks_per_seq, float softmax_scale, float skip_threshold,
                                     void* workspace, size_t workspace_bytes, float* out, tq_stream_t stream) {
  if (!ctx || !q || !out || !seq_lens || !k_views || !v_views || !k_view_layers || !v_view_layers)
    return TQ_ERR_INVALID_ARG;
  if (n_layers < 0 || batch < 0 || n_q_heads < 1 || max_ctx < 0) return TQ_ERR_INVALID_ARG;
  if (q_is_fp16 != 0 && q_is_fp16 != 1) return TQ_ERR_INVALID_ARG;
  if (!std::isfinite(softmax_scale) || !(skip_threshold >= 0.0f) || !std::isfinite(skip_threshold))
    return TQ_ERR_INVALID_ARG;
  if (n_layers > 65535) return TQ_ERR_UNSUPPORTED;  // layer maps hold 16-bit indices
  const int d = ctx->d;
  int H = 0;
  for (int l = 0; l < n_layers; ++l) {  // every layer validated before anything is launched
    DevView kd{}, vd{};
    if (!layer_view(&k_views[l], k_view_layers[l], 1, &kd) || !layer_view(&v_views[l], v_view_layers[l], 1, &vd))
      return TQ_ERR_INVALID_ARG;
    if (k_view_layers[l] > 65535 || v_view_layers[l] > 65535) return TQ_ERR_UNSUPPORTED;
    if (kd.d != d || vd.d != d || kd.H != vd.H || (l > 0 && kd.H != H)) return TQ_ERR_INVALID_ARG;
    H = kd.H;
    if (kd.page_size != vd.page_size || kd.num_pages != vd.num_pages) return TQ_ERR_INVALID_ARG;
    const bool k_ok = format_is_turbo(kd.format) || kd.format == TQ_FMT_Q8_0;
    const bool v_ok = (format_is_turbo(vd.format) && !vd.has_qjl) || vd.format == TQ_FMT_Q8_0;
    if (!k_ok || !v_ok) return TQ_ERR_UNSUPPORTED;
    if (block_table) {
      if (max_blocks_per_seq < 1 || (int64_t)max_blocks_per_seq * kd.page_size < max_ctx) return TQ_ERR_INVALID_ARG;
    } else if (max_ctx > kd.page_size || batch > kd.num_pages) {
      return TQ_ERR_INVALID_ARG;
    }
  }
  if (n_layers == 0 || batch == 0) return TQ_OK;
  if (n_q_heads % H != 0 || n_q_heads / H > 16) return TQ_ERR_UNSUPPORTED;
  // one plan for the whole call, so the workspace of tq_decode_workspace_bytes(n_layers, ...) holds every run
  const DecodePlan plan = plan_decode(ctx->sm_count, d, n_layers, batch, n_q_heads, max_ctx);
  if (!workspace || workspace_bytes < plan.bytes || (reinterpret_cast<uintptr_t>(workspace) & 255))
    return TQ_ERR_WORKSPACE;
  // layers grouped by their (K view, V view) pair, in order of first appearance; one launch set per
  // group (at most DecodeArgs::kMapMax layers each) with a layer map
  std::vector<int> done(n_layers, 0);
  for (int l0 = 0; l0 < n_layers; ++l0) {
    if (done[l0]) continue;
    std::vector<int> group;
    for (int l = l0; l < n_layers; ++l)
      if (!done[l] && same_view(k_views[l], k_views[l0]) && same_view(v_views[l], v_views[l0])) {
        group.push_back(l);
        done[l] = 1;
      }
    for (size_t c0 = 0; c0 < group.size(); c0 += DecodeArgs::kMapMax) {
      const int cnt = (int)std::min(group.size() - c0, (size_t)DecodeArgs::kMapMax);
      DecodeArgs a{};
      make_dev_view(&k_views[l0], &a.k);
      make_dev_view(&v_views[l0], &a.v);
      a.n_map = cnt;
      for (int i = 0; i < cnt; ++i) {
        const int l = group[c0 + i];
        a.k_layer[i] = (uint16_t)k_view_layers[l];
        a.v_layer[i] = (uint16_t)v_view_layers[l];
        a.q_layer[i] = (uint16_t)l;
      }
      a.q = q;
      a.q_is_fp16 = q_is_fp16;
      a.n_layers = cnt;
      a.batch = batch;
      a.n_q_heads = n_q_heads;
      a.layer_begin = 0;
      a.seq_lens = seq_lens;
      a.max_ctx = max_ctx;
      a.block_table = block_table;
      a.max_blocks_per_seq = block_table ? max_blocks_per_seq : 1;
      a.softmax_scale = softmax_scale;
      a.skip_threshold = skip_threshold;
      a.out = out;
      // the group's own split plan when it fits in the workspace (a few boundary layers want shorter
      // splits than the whole call to fill the GPU), else the whole call's splits for its rows only
      DecodePlan rp = plan_decode(ctx->sm_count, d, cnt, batch, n_q_heads, max_ctx);
      if (rp.bytes > workspace_bytes) {
        rp = plan;
        const size_t rows = (size_t)cnt * batch * n_q_heads;
        rp.qprep_floats = rows * 2 * d;
        rp.partial_floats = rows * plan.n_splits * (d + 4);
      }
      const tq_status st = cuda_status(
          launch_decode(ctx->tables, a, rp, workspace, ctx->sm_count, reinterpret_cast<cudaStream_t>(stream)));
      if (st != TQ_OK) return st;
    }
  }
  return TQ_OK;
}

// ---------------------------------------------------------------------------
// chunked-prefill attention
// ---------------------------------------------------------------------------

size_t tq_prefill_workspace_bytes(const tq_context* ctx, int n_tokens, int n_q_heads) {
  if (!ctx || n_tokens < 0 || n_q_heads < 1) return 0;
  return prefill_workspace(n_tokens, n_q_heads, ctx->d);
}

tq_status tq_prefill_attention(const tq_context* ctx, const void* q, int q_is_fp16, int n_tokens, int n_q_heads,
                               const tq_cache_view* k_view, const tq_cache_view* v_view, int layer, int seq,
                               const int32_t* block_table, int max_blocks, int start, float softmax_scale,
                               void* workspace, size_t workspace_bytes, float* out, tq_stream_t stream) {
  if (!ctx || !q || !out || !k_view || !v_view) return TQ_ERR_INVALID_ARG;
  if (q_is_fp16 != 0 && q_is_fp16 != 1) return TQ_ERR_INVALID_ARG;
  if (n_tokens < 0 || n_q_heads < 1 || start < 0 || layer < 0 || !std::isfinite(softmax_scale))
    return TQ_ERR_INVALID_ARG;
  DevView k{}, v{};
  if (!make_dev_view(k_view, &k) || !make_dev_view(v_view, &v)) return TQ_ERR_INVALID_ARG;
  if (k.d != ctx->d || v.d != ctx->d || k.H != v.H || k.page_size != v.page_size || k.num_pages != v.num_pages)
    return TQ_ERR_INVALID_ARG;
  if (layer >= k.n_layers || layer >= v.n_layers) return TQ_ERR_INVALID_ARG;
  if (ctx->d != 128) return TQ_ERR_UNSUPPORTED;
  if (!(format_is_turbo(k.format) && k.has_qjl) || !(format_is_turbo(v.format) && !v.has_qjl))
    return TQ_ERR_UNSUPPORTED;  // turbo K with its QJL stage, turbo-MSE V
  if (n_q_heads % k.H != 0) return TQ_ERR_UNSUPPORTED;
  const long long keys = (long long)start + n_tokens;
  if (block_table) {
    if (max_blocks < 1 || (long long)max_blocks * k.page_size < keys) return TQ_ERR_INVALID_ARG;
  } else if (seq < 0 || seq >= k.num_pages || keys > k.page_size) {
    return TQ_ERR_INVALID_ARG;  // contiguous: sequence seq is page seq of capacity page_size
  }
  if (keys >= (1LL << 31) || (long long)n_tokens * n_q_heads >= (1LL << 31)) return TQ_ERR_UNSUPPORTED;
  if (n_tokens == 0) return TQ_OK;
  if (!workspace || workspace_bytes < prefill_workspace(n_tokens, n_q_heads, ctx->d) ||
      (reinterpret_cast<uintptr_t>(workspace) & 255))
    return TQ_ERR_WORKSPACE;
  DecodeArgs qa{};
  qa.q = q;
  qa.q_is_fp16 = q_is_fp16;
  qa.n_layers = 1;
  qa.batch = n_tokens;
  qa.n_q_heads = n_q_heads;
  qa.k = k;
  qa.v = v;
  qa.softmax_scale = softmax_scale;
  qa.out = out;
  return cuda_status(launch_prefill(ctx->tables, qa, k, v, layer, seq, block_table, max_blocks, start,
                                    ctx->f16_scale_h[k.idx_bits - 1], ctx->f16_scale_h[v.idx_bits - 1], workspace,
                                    reinterpret_cast<cudaStream_t>(stream)));
}

}  // extern "C"
