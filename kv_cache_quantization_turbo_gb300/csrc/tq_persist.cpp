// Persistence of a compressed cache: a cache view written to a file and read back.
//
// Out of the hot path.  The source pages save a compressed cache to disk as arrays plus a small
// metadata file ("mac-code TurboQuant analysis", section 2.4: an .npz of the arrays and a
// .meta.json beside it); here it is one self-describing file:
//
//   "TQCACHE1\n"
//   one JSON object on one line, then "\n": format, geometry, byte counts, the context's seeds,
//     a hash of the context's tables (signs, QJL matrix, codebooks) and a hash of the data
//   zero padding up to the next multiple of 4096 bytes
//   the payload array (every layer of the view), then the header array
//
// The arrays are the view's own bytes, in the view's order ([layer][page][head][slot] vectors), so
// a file is read back into a view of the same geometry and format only, made with the same tables
// (the codes mean nothing without them).  Device arrays go through a host buffer of at most
// 64 MiB; host arrays (host_memory = 1) are read and written directly.
#include <cinttypes>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <string>

#include "tq_internal.h"

namespace {

constexpr char kMagic[] = "TQCACHE1\n";
constexpr size_t kAlign = 4096;
constexpr size_t kChunk = size_t(64) << 20;

// FNV-1a, 64-bit (Fowler, Noll, Vo), taken over little-endian 64-bit words of each block passed
// to add (and its trailing bytes one at a time), so that gigabytes hash at memory speed.  Save and
// load pass the same blocks (arrays in 64 MiB chunks), so they agree.
struct Fnv {
  uint64_t h = 0xcbf29ce484222325ull;
  void add(const void* p, size_t n) {
    const unsigned char* b = static_cast<const unsigned char*>(p);
    size_t i = 0;
    for (; i + 8 <= n; i += 8) {
      uint64_t w = 0;
      for (int k = 0; k < 8; ++k) w |= (uint64_t)b[i + k] << (8 * k);
      h ^= w;
      h *= 0x100000001b3ull;
    }
    for (; i < n; ++i) {
      h ^= b[i];
      h *= 0x100000001b3ull;
    }
  }
};

uint64_t tables_hash(const tq_context* ctx) {
  Fnv f;
  const int32_t d = ctx->d;
  f.add(&d, sizeof(d));
  f.add(ctx->signs_h, (size_t)d);
  f.add(ctx->S_h, sizeof(float) * (size_t)d * d);
  f.add(ctx->centroids_h, sizeof(ctx->centroids_h));
  f.add(ctx->boundaries_h, sizeof(ctx->boundaries_h));
  return f.h;
}

struct Geometry {
  size_t pay_bytes, hdr_bytes;  // whole arrays
};

bool geometry(const tq_cache_view* v, Geometry* g) {
  if (!v || v->head_dim < 1 || v->n_kv_heads < 1 || v->page_size < 1 || v->num_pages < 1 || v->n_layers < 1)
    return false;
  const size_t pb = tq_payload_bytes((tq_format)v->format, v->head_dim, v->bits);
  const size_t hb = tq_header_bytes((tq_format)v->format, v->head_dim, v->bits);
  if (pb == 0 || hb == 0) return false;
  const size_t n = (size_t)v->n_layers * (size_t)v->num_pages * (size_t)v->n_kv_heads * (size_t)v->page_size;
  g->pay_bytes = n * pb;
  g->hdr_bytes = n * hb;
  return true;
}

std::string header_json(const tq_cache_view* v, const Geometry& g, const tq_context* ctx, uint64_t data_hash) {
  char buf[1024];
  std::snprintf(buf, sizeof(buf),
                "{\"version\": 1, \"format\": \"%s\", \"format_id\": %d, \"head_dim\": %d, \"n_kv_heads\": %d, "
                "\"page_size\": %d, \"num_pages\": %" PRId64 ", \"n_layers\": %d, \"bits\": %d, "
                "\"payload_bytes\": %zu, \"header_bytes\": %zu, \"wht_seed\": %u, \"qjl_seed\": %u, "
                "\"tables_hash\": \"%016" PRIx64 "\", \"data_hash\": \"%016" PRIx64 "\", "
                "\"layout\": \"vectors [n_layers][num_pages][n_kv_heads][page_size]; payload array, then header "
                "array\"}",
                tq_format_name((tq_format)v->format), v->format, v->head_dim, v->n_kv_heads, v->page_size,
                (int64_t)v->num_pages, v->n_layers, v->format == TQ_FMT_MINMAX ? v->bits : 0, g.pay_bytes,
                g.hdr_bytes, ctx ? ctx->wht_seed : 0u, ctx ? ctx->qjl_seed : 0u, ctx ? tables_hash(ctx) : 0ull,
                data_hash);
  return std::string(buf);
}

// Value of "key": number (or "0x..."-less hex string when hex) in a one-line JSON object we wrote.
bool json_int(const std::string& js, const char* key, int64_t* out) {
  const std::string k = std::string("\"") + key + "\": ";
  const size_t p = js.find(k);
  if (p == std::string::npos) return false;
  char* end = nullptr;
  const long long v = std::strtoll(js.c_str() + p + k.size(), &end, 10);
  if (end == js.c_str() + p + k.size()) return false;
  *out = v;
  return true;
}
bool json_hex(const std::string& js, const char* key, uint64_t* out) {
  const std::string k = std::string("\"") + key + "\": \"";
  const size_t p = js.find(k);
  if (p == std::string::npos) return false;
  char* end = nullptr;
  const unsigned long long v = std::strtoull(js.c_str() + p + k.size(), &end, 16);
  if (end != js.c_str() + p + k.size() + 16) return false;
  *out = v;
  return true;
}

struct File {
  FILE* f = nullptr;
  ~File() {
    if (f) std::fclose(f);
  }
};

// Reads the magic line and the JSON line; leaves the stream at the first data byte.
tq_status read_header(FILE* f, std::string* js, size_t* data_offset) {
  char magic[sizeof(kMagic) - 1];
  if (std::fread(magic, 1, sizeof(magic), f) != sizeof(magic) || std::memcmp(magic, kMagic, sizeof(magic)) != 0)
    return TQ_ERR_INVALID_ARG;
  js->clear();
  for (;;) {
    const int c = std::fgetc(f);
    if (c == EOF || js->size() > 65536) return TQ_ERR_INVALID_ARG;
    if (c == '\n') break;
    js->push_back((char)c);
  }
  const size_t used = sizeof(kMagic) - 1 + js->size() + 1;
  *data_offset = (used + kAlign - 1) / kAlign * kAlign;
  if (std::fseek(f, (long)*data_offset, SEEK_SET) != 0) return TQ_ERR_INVALID_ARG;
  return TQ_OK;
}

// Moves n bytes between a file and an array (device or host), hashing them.
tq_status stream_array(FILE* f, void* arr, size_t n, bool host, bool writing, Fnv* h) {
  unsigned char* a = static_cast<unsigned char*>(arr);
  unsigned char* bounce = nullptr;
  if (!host) {
    bounce = static_cast<unsigned char*>(std::malloc(n < kChunk ? (n ? n : 1) : kChunk));
    if (!bounce) return TQ_ERR_OOM;
  }
  tq_status st = TQ_OK;
  for (size_t off = 0; off < n && st == TQ_OK;) {
    const size_t m = n - off < kChunk ? n - off : kChunk;
    unsigned char* hp = host ? a + off : bounce;
    if (writing) {
      if (!host && cudaMemcpy(hp, a + off, m, cudaMemcpyDeviceToHost) != cudaSuccess) st = TQ_ERR_CUDA;
      if (st == TQ_OK) {
        h->add(hp, m);
        if (std::fwrite(hp, 1, m, f) != m) st = TQ_ERR_INVALID_ARG;
      }
    } else {
      if (std::fread(hp, 1, m, f) != m) st = TQ_ERR_INVALID_ARG;
      if (st == TQ_OK) {
        h->add(hp, m);
        if (!host && cudaMemcpy(a + off, hp, m, cudaMemcpyHostToDevice) != cudaSuccess) st = TQ_ERR_CUDA;
      }
    }
    off += m;
  }
  std::free(bounce);
  return st;
}

}  // namespace

extern "C" {

tq_status tq_context_tables_hash(const tq_context* ctx, uint64_t* hash) {
  if (!ctx || !hash) return TQ_ERR_INVALID_ARG;
  *hash = tables_hash(ctx);
  return TQ_OK;
}

tq_status tq_cache_save(const tq_context* ctx, const tq_cache_view* view, int host_memory, const char* path) {
  Geometry g;
  if (!path || !geometry(view, &g) || !view->payload || !view->header || (host_memory != 0 && host_memory != 1))
    return TQ_ERR_INVALID_ARG;
  if (ctx && ctx->d != view->head_dim) return TQ_ERR_INVALID_ARG;
  if (!host_memory && cudaDeviceSynchronize() != cudaSuccess) return TQ_ERR_CUDA;
  // The data hash goes into the JSON line, which precedes the data: write the data first at its
  // offset (computed from a JSON line of the final length: the hash field has a fixed width).
  const std::string probe = header_json(view, g, ctx, 0);
  const size_t used = sizeof(kMagic) - 1 + probe.size() + 1;
  const size_t data_offset = (used + kAlign - 1) / kAlign * kAlign;
  const std::string tmp = std::string(path) + ".partial";
  File out;
  out.f = std::fopen(tmp.c_str(), "wb");
  if (!out.f) return TQ_ERR_INVALID_ARG;
  if (std::fseek(out.f, (long)data_offset, SEEK_SET) != 0) return TQ_ERR_INVALID_ARG;
  Fnv h;
  tq_status st = stream_array(out.f, view->payload, g.pay_bytes, host_memory, true, &h);
  if (st == TQ_OK) st = stream_array(out.f, view->header, g.hdr_bytes, host_memory, true, &h);
  if (st != TQ_OK) return st;
  const std::string js = header_json(view, g, ctx, h.h);
  std::string head(kMagic);
  head += js;
  head += '\n';
  head.resize(data_offset, '\0');
  if (std::fseek(out.f, 0, SEEK_SET) != 0 || std::fwrite(head.data(), 1, head.size(), out.f) != head.size())
    return TQ_ERR_INVALID_ARG;
  if (std::fclose(out.f) != 0) {
    out.f = nullptr;
    return TQ_ERR_INVALID_ARG;
  }
  out.f = nullptr;
  return std::rename(tmp.c_str(), path) == 0 ? TQ_OK : TQ_ERR_INVALID_ARG;
}

tq_status tq_cache_file_info(const char* path, tq_cache_view* geometry_out, uint64_t* tables_hash_out) {
  if (!path || !geometry_out) return TQ_ERR_INVALID_ARG;
  File in;
  in.f = std::fopen(path, "rb");
  if (!in.f) return TQ_ERR_INVALID_ARG;
  std::string js;
  size_t off = 0;
  if (read_header(in.f, &js, &off) != TQ_OK) return TQ_ERR_INVALID_ARG;
  int64_t fmt, d, H, P, pages, L, bits;
  uint64_t th;
  if (!json_int(js, "format_id", &fmt) || !json_int(js, "head_dim", &d) || !json_int(js, "n_kv_heads", &H) ||
      !json_int(js, "page_size", &P) || !json_int(js, "num_pages", &pages) || !json_int(js, "n_layers", &L) ||
      !json_int(js, "bits", &bits) || !json_hex(js, "tables_hash", &th))
    return TQ_ERR_INVALID_ARG;
  tq_cache_view v{};
  v.format = (int32_t)fmt;
  v.head_dim = (int32_t)d;
  v.n_kv_heads = (int32_t)H;
  v.page_size = (int32_t)P;
  v.num_pages = pages;
  v.n_layers = (int32_t)L;
  v.bits = (int32_t)bits;
  Geometry g;
  if (!geometry(&v, &g)) return TQ_ERR_INVALID_ARG;
  *geometry_out = v;
  if (tables_hash_out) *tables_hash_out = th;
  return TQ_OK;
}

tq_status tq_cache_load(const tq_context* ctx, const tq_cache_view* view, int host_memory, const char* path) {
  Geometry g;
  if (!path || !geometry(view, &g) || !view->payload || !view->header || (host_memory != 0 && host_memory != 1))
    return TQ_ERR_INVALID_ARG;
  tq_cache_view fv{};
  uint64_t th = 0;
  if (tq_cache_file_info(path, &fv, &th) != TQ_OK) return TQ_ERR_INVALID_ARG;
  const int vbits = view->format == TQ_FMT_MINMAX ? view->bits : 0;
  if (fv.format != view->format || fv.head_dim != view->head_dim || fv.n_kv_heads != view->n_kv_heads ||
      fv.page_size != view->page_size || fv.num_pages != view->num_pages || fv.n_layers != view->n_layers ||
      fv.bits != vbits)
    return TQ_ERR_INVALID_ARG;
  if (ctx && (ctx->d != view->head_dim || th != tables_hash(ctx))) return TQ_ERR_INVALID_ARG;
  File in;
  in.f = std::fopen(path, "rb");
  if (!in.f) return TQ_ERR_INVALID_ARG;
  std::string js;
  size_t off = 0;
  if (read_header(in.f, &js, &off) != TQ_OK) return TQ_ERR_INVALID_ARG;
  int64_t pay = -1, hdr = -1;
  uint64_t want = 0;
  if (!json_int(js, "payload_bytes", &pay) || !json_int(js, "header_bytes", &hdr) ||
      !json_hex(js, "data_hash", &want) || (size_t)pay != g.pay_bytes || (size_t)hdr != g.hdr_bytes)
    return TQ_ERR_INVALID_ARG;
  if (!host_memory && cudaDeviceSynchronize() != cudaSuccess) return TQ_ERR_CUDA;
  Fnv h;
  tq_status st = stream_array(in.f, view->payload, g.pay_bytes, host_memory, false, &h);
  if (st == TQ_OK) st = stream_array(in.f, view->header, g.hdr_bytes, host_memory, false, &h);
  if (st != TQ_OK) return st;
  if (std::fgetc(in.f) != EOF) return TQ_ERR_INVALID_ARG;  // trailing bytes
  return h.h == want ? TQ_OK : TQ_ERR_INVALID_ARG;
}

}  // extern "C"
