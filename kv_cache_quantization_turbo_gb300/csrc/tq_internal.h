// Internal declarations shared by the host API (tq_api.cpp) and the CUDA
// translation units.  Not part of the public ABI (see include/tq.h).
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "../../include/tq.h"

namespace tq {

// Status-word bits written by kernels (documented in tq_get_status).
enum : uint32_t { kFlagSeqLen = 1u, kFlagBlockTable = 2u, kFlagSlot = 4u, kFlagTimeout = 8u };

// Highest supported head_dim and codebook sizes.
constexpr int kMaxDim = 256;
constexpr int kMaxLevels = 8;  // turbo stage 1 uses at most 3 bits

// Plain-old-data description of a cache view, passed by value to kernels.
struct DevView {
  int format;       // tq_format
  int d;            // head_dim
  int H;            // n_kv_heads
  int page_size;
  long long num_pages;
  int n_layers;
  int idx_bits;     // stage-1 index bits (turbo), or minmax bits, or 8 (q8_0)
  int code_bits;    // bits per coordinate in the payload (turbo K: idx_bits + 1)
  int has_qjl;      // turbo K formats
  int pay_bytes;    // payload bytes per vector
  int hdr_bytes;    // header bytes per vector
  unsigned char* payload;
  unsigned char* header;
};

// Device tables owned by a context.
struct DevTables {
  int d;
  const int8_t* signs;       // [d]
  const float* S;            // [d][d], row j = projection j
  const float* S_T;          // [d][d], S_T[i][j] = S[j][i]
  // S split into high and low fp16 parts (S = hi + lo to ~22 bits) in mma.sync m16n8k16
  // B-fragment order: entry ((nb * d/16 + ks) * 32 + lane) = {hi(b0), hi(b1), lo(b0), lo(b1)}
  // with b0 = S[8nb + lane/4][16ks + 2(lane%4) + {0,1}], b1 = the same at + 8 coordinates
  const uint4* S_frag;
  const float* centroids;    // [3][8]  (bits 1, 2, 3)
  const float* boundaries;   // [3][7]
  const float* f16_scale;    // [3]: lambda per bit width, so that lambda * centroid is (nearly) an fp16 value
  uint32_t* status;          // device status word
};

bool format_is_turbo(int f);
bool format_has_qjl(int f);
int format_idx_bits(int f, int minmax_bits);

// Fills a DevView from a public view; returns false if the view is invalid.
bool make_dev_view(const tq_cache_view* v, DevView* out);

// ---- launchers (defined in the .cu files); all return cudaGetLastError() ----
cudaError_t launch_encode(const DevTables& t, const DevView& view, const __half* x, int layer_begin,
                          int n_layers, int n_tokens, long long layer_stride, long long token_stride,
                          const long long* slots, long long slot_begin, int sm_count, cudaStream_t s);

cudaError_t launch_dequant(const DevTables& t, const DevView& view, int layer, const long long* slots,
                           long long slot_begin, int n, int include_qjl, float* out, cudaStream_t s);

struct DecodeArgs {
  const void* q;
  int q_is_fp16;
  int n_layers, batch, n_q_heads;
  DevView k, v;
  int layer_begin;
  const int32_t* seq_lens;
  int max_ctx;
  const int32_t* block_table;
  int max_blocks_per_seq;
  float softmax_scale, skip_threshold;
  float* out;
  // Layer map of a launch over layers that are not consecutive in their views (per-layer views):
  // launch layer i reads layer k_layer[i] of the K view, v_layer[i] of the V view, and query and
  // output layer q_layer[i].  n_map = 0: layer_begin + i in both views, i for q and out.
  static constexpr int kMapMax = 128;
  int n_map;
  uint16_t k_layer[kMapMax], v_layer[kMapMax], q_layer[kMapMax];
};

__host__ __device__ __forceinline__ int k_layer_of(const DecodeArgs& a, int i) {
  return a.n_map ? (int)a.k_layer[i] : a.layer_begin + i;
}
__host__ __device__ __forceinline__ int v_layer_of(const DecodeArgs& a, int i) {
  return a.n_map ? (int)a.v_layer[i] : a.layer_begin + i;
}
// Row of q / out for launch row `row` = (launch layer, sequence, query head).
__host__ __device__ __forceinline__ long long io_row_of(const DecodeArgs& a, long long row) {
  if (!a.n_map) return row;
  const long long per_layer = (long long)a.batch * a.n_q_heads;
  const long long i = row / per_layer;
  return (long long)a.q_layer[i] * per_layer + (row - i * per_layer);
}

// Split-K plan for a decode call: tokens per split and the number of splits.
struct DecodePlan {
  int split_tokens;
  int n_splits;
  size_t partial_floats;   // floats of split-K partials
  size_t qprep_floats;     // floats of prepared queries
  size_t bytes;            // total workspace bytes (256-byte aligned parts)
};
DecodePlan plan_decode(int sm_count, int d, int n_layers, int batch, int n_q_heads, int max_ctx);

// The decode prologue (q' = scale H diag(s) q, S q') for the rows of a: writes qprep [rows][2d]
// and zeroes counter[0..1].  Shared by the prefill attention.
cudaError_t launch_qprep(const DevTables& t, const DecodeArgs& a, float* qprep, unsigned int* counter,
                         cudaStream_t s);

// Chunked-prefill attention (tq_prefill.cu), head_dim 128, turbo K and turbo-MSE V: the rows of qa
// (batch = chunk tokens, n_layers = 1) against layer `layer` of k and v; lam_k / lam_v are the
// fp16 table scales of the K and V index widths.
size_t prefill_workspace(int n_tokens, int n_q_heads, int d);
cudaError_t launch_prefill(const DevTables& t, const DecodeArgs& qa, const DevView& k, const DevView& v, int layer,
                           int seq, const int32_t* block_table, int max_blocks, int start, float lam_k, float lam_v,
                           void* workspace, cudaStream_t s);

cudaError_t launch_decode(const DevTables& t, const DecodeArgs& a, const DecodePlan& plan,
                          void* workspace, int sm_count, cudaStream_t s);

// Everything the decode kernels receive (by value).
struct DecodeLaunch {
  DecodeArgs a;
  DevTables tab;
  int split_tokens, n_splits, G;
  int g_off, g_cnt;  // tensor-core kernel: query heads [g_off, g_off + g_cnt) of each KV head's G
  int g_halves;      // 2: every work item runs twice, on heads [0, g_cnt) and [g_cnt, G) (9 to 16 heads)
  float* qprep;    // [rows][2d]: q' then Sq'
  float* partial;  // [rows][n_splits][d + 4]: m (natural log units), l, -, -, acc[d]
  unsigned int* counter;  // two work-item counters (zeroed by the prologue kernel)
  int keep_partials;      // 1: the partials are stored evict-last in L2 (they fit beside the streamed cache)
};
// Partials up to this size are kept in L2 (evict-last) until the combine reads them; larger sets
// would crowd the cache tiles that the attention kernel prefetches into the 126 MB L2.
constexpr size_t kKeepPartialsMaxBytes = 40u << 20;

// Split-K attention on tensor cores (tq_decode_mma.cuh), parameterised by the formats: K code width wk
// (q8_0 = 0, turbo K = index bits + 1), V code width wv (q8_0 = 0, turbo-MSE V = index bits),
// one translation unit per head_dim.
bool mma_has_d64(int wk, int wv);
bool mma_has_d128(int wk, int wv);
bool mma_has_d256(int wk, int wv);
cudaError_t mma_launch_d64(const DecodeLaunch& k, int wk, int wv, int sm_count, cudaStream_t s);
cudaError_t mma_launch_d128(const DecodeLaunch& k, int wk, int wv, int sm_count, cudaStream_t s);
cudaError_t mma_launch_d256(const DecodeLaunch& k, int wk, int wv, int sm_count, cudaStream_t s);

}  // namespace tq

struct tq_context {
  int device;
  int d;
  int sm_count;
  uint32_t wht_seed, qjl_seed;  // as given at creation (informational when the tables were passed in)
  // host copies
  int8_t signs_h[tq::kMaxDim];
  float centroids_h[3][8];
  float boundaries_h[3][7];
  float f16_scale_h[3];
  float* S_h;  // [d*d]
  // device allocations
  void* dev_block;  // one allocation holding every table
  tq::DevTables tables;
};
