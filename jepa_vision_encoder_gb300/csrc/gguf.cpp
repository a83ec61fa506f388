// gguf.cpp -- a GGUF (v2 / v3) reader for encoder files, with the loader's checks of the jepa.cpp
// pages ("Architecture", Robustness: what the loader validates). Every count, length, offset and
// extent read from the file is checked against the file before it is used; nothing is clamped or
// defaulted silently. Host code only.
//
// Layout (the GGUF format): magic "GGUF", u32 version, u64 tensor count, u64 key/value count; the
// key/value pairs (string key, u32 value type, value); the tensor infos (string name, u32 n_dims,
// u64 dims[n_dims] (ggml order: dims[0] is the innermost, PyTorch's last), u32 ggml type, u64
// offset into the data section); padding to general.alignment (32 by default); the data section.
#include <cmath>
#include <cstdio>
#include <cstring>
#include <limits>
#include <string>
#include <vector>

#include "internal.h"
#include "jepa.h"
#include "jepa_synth.h"

namespace jepa {
namespace {

constexpr uint64_t kMaxString = 1ull << 20, kMaxKv = 1ull << 16, kMaxTensors = 1ull << 20, kMaxArray = 1ull << 24;

enum : uint32_t { kU8 = 0, kI8, kU16, kI16, kU32, kI32, kF32, kBool, kString, kArray, kU64, kI64, kF64 };

// ggml tensor types this reader knows the storage of: block size and bytes per block.
struct TypeInfo {
  uint32_t type, block, bytes;
  const char* name;
};
const TypeInfo kTypes[] = {
    {0, 1, 4, "f32"},     {1, 1, 2, "f16"},     {2, 32, 18, "q4_0"},   {3, 32, 20, "q4_1"},   {6, 32, 22, "q5_0"},
    {7, 32, 24, "q5_1"},  {8, 32, 34, "q8_0"},  {9, 32, 36, "q8_1"},   {10, 256, 84, "q2_k"}, {11, 256, 110, "q3_k"},
    {12, 256, 144, "q4_k"}, {13, 256, 176, "q5_k"}, {14, 256, 210, "q6_k"}, {15, 256, 292, "q8_k"},
    {30, 1, 2, "bf16"}};
const TypeInfo* type_info(uint32_t t) {
  for (const auto& i : kTypes)
    if (i.type == t) return &i;
  return nullptr;
}

struct Reader {
  FILE* f = nullptr;
  uint64_t size = 0, pos = 0;
  bool read(void* dst, uint64_t n) {
    if (pos > size || n > size - pos) return false;
    if (n && fread(dst, 1, n, f) != n) return false;
    pos += n;
    return true;
  }
  bool skip(uint64_t n) {
    if (pos > size || n > size - pos) return false;
    pos += n;
    return fseeko(f, (off_t)pos, SEEK_SET) == 0;
  }
  template <class T>
  bool get(T* v) { return read(v, sizeof(T)); }
  bool str(std::string* s) {
    uint64_t n = 0;
    if (!get(&n) || n > kMaxString || pos > size || n > size - pos) return false;
    s->resize(n);
    return read(s->data(), n);
  }
};

uint64_t scalar_bytes(uint32_t t) {
  switch (t) {
    case kU8: case kI8: case kBool: return 1;
    case kU16: case kI16: return 2;
    case kU32: case kI32: case kF32: return 4;
    case kU64: case kI64: case kF64: return 8;
    default: return 0;
  }
}

bool read_value(Reader& r, uint32_t type, GgufValue* v, int depth) {
  v->type = type;
  switch (type) {
    case kU8: { uint8_t x; if (!r.get(&x)) return false; v->u = x; v->i = x; v->f = x; return true; }
    case kI8: { int8_t x; if (!r.get(&x)) return false; v->i = x; v->f = x; v->u = (uint64_t)x; return true; }
    case kU16: { uint16_t x; if (!r.get(&x)) return false; v->u = x; v->i = x; v->f = x; return true; }
    case kI16: { int16_t x; if (!r.get(&x)) return false; v->i = x; v->f = x; v->u = (uint64_t)x; return true; }
    case kU32: { uint32_t x; if (!r.get(&x)) return false; v->u = x; v->i = x; v->f = x; return true; }
    case kI32: { int32_t x; if (!r.get(&x)) return false; v->i = x; v->f = x; v->u = (uint64_t)x; return true; }
    case kU64: { uint64_t x; if (!r.get(&x)) return false; v->u = x; v->i = (int64_t)x; v->f = (double)x; return true; }
    case kI64: { int64_t x; if (!r.get(&x)) return false; v->i = x; v->f = (double)x; v->u = (uint64_t)x; return true; }
    case kF32: { float x; if (!r.get(&x)) return false; v->f = x; return true; }
    case kF64: { double x; if (!r.get(&x)) return false; v->f = x; return true; }
    case kBool: { uint8_t x; if (!r.get(&x) || x > 1) return false; v->u = x; v->i = x; return true; }
    case kString: return r.str(&v->s);
    case kArray: {
      if (depth > 0) return false;  // nested arrays: not part of any jepa key
      uint32_t et = 0;
      uint64_t n = 0;
      if (!r.get(&et) || !r.get(&n) || n > kMaxArray) return false;
      v->array_type = et;
      v->array_len = n;
      if (et == kString) {
        for (uint64_t i = 0; i < n; ++i) {
          GgufValue e;
          if (!read_value(r, kString, &e, depth + 1)) return false;
        }
        return true;
      }
      const uint64_t eb = scalar_bytes(et);
      if (!eb || n > (r.size - r.pos) / eb) return false;
      if (et == kF32 || et == kF64) return r.skip(n * eb);
      v->ints.reserve((size_t)n);
      for (uint64_t i = 0; i < n; ++i) {
        GgufValue e;
        if (!read_value(r, et, &e, depth + 1)) return false;
        v->ints.push_back(e.i);
      }
      return true;
    }
    default: return false;
  }
}

struct FileCloser {
  FILE* f;
  ~FileCloser() {
    if (f) fclose(f);
  }
};
}  // namespace

const GgufValue* GgufFile::get(const std::string& key) const {
  for (const auto& kv : kvs)
    if (kv.first == key) return &kv.second;
  return nullptr;
}

const GgufTensor* GgufFile::find(const std::string& name) const {
  for (const auto& t : tensors)
    if (t.name == name) return &t;
  return nullptr;
}

jepa_status gguf_open(const char* path, GgufFile* g) {
  if (!path || !g) return fail(JEPA_E_INVALID_ARG, "gguf: null argument");
  FILE* f = fopen(path, "rb");
  if (!f) return fail(JEPA_E_INVALID_ARG, "gguf: cannot open '%s'", path);
  FileCloser closer{f};
  if (fseeko(f, 0, SEEK_END) != 0) return fail(JEPA_E_INVALID_ARG, "gguf: cannot seek '%s'", path);
  const off_t end = ftello(f);
  if (end < 0 || fseeko(f, 0, SEEK_SET) != 0) return fail(JEPA_E_INVALID_ARG, "gguf: cannot size '%s'", path);
  Reader r;
  r.f = f;
  r.size = (uint64_t)end;
  g->path = path;
  g->file_size = r.size;
  char magic[4];
  if (!r.read(magic, 4) || memcmp(magic, "GGUF", 4) != 0) return fail(JEPA_E_INVALID_ARG, "gguf: '%s' is not a GGUF file", path);
  uint64_t n_tensors = 0, n_kv = 0;
  if (!r.get(&g->version)) return fail(JEPA_E_INVALID_ARG, "gguf: truncated header");
  if (g->version != 2 && g->version != 3) return fail(JEPA_E_INVALID_ARG, "gguf: version %u (2 or 3 expected)", g->version);
  if (!r.get(&n_tensors) || !r.get(&n_kv)) return fail(JEPA_E_INVALID_ARG, "gguf: truncated header");
  if (n_tensors > kMaxTensors || n_kv > kMaxKv)
    return fail(JEPA_E_INVALID_ARG, "gguf: %llu tensors / %llu keys out of range", (unsigned long long)n_tensors,
                (unsigned long long)n_kv);
  for (uint64_t i = 0; i < n_kv; ++i) {
    std::string key;
    uint32_t type = 0;
    GgufValue v;
    if (!r.str(&key) || !r.get(&type) || !read_value(r, type, &v, 0))
      return fail(JEPA_E_INVALID_ARG, "gguf: key/value %llu malformed or truncated", (unsigned long long)i);
    if (g->get(key)) return fail(JEPA_E_INVALID_ARG, "gguf: key '%s' appears twice", key.c_str());
    g->kvs.emplace_back(key, v);
  }
  g->alignment = 32;
  if (const GgufValue* a = g->get("general.alignment")) {
    if (a->type != kU32 || a->u == 0 || a->u > 65536 || (a->u & (a->u - 1)))
      return fail(JEPA_E_INVALID_ARG, "gguf: general.alignment must be a u32 power of two up to 65536");
    g->alignment = (uint32_t)a->u;
  }
  for (uint64_t i = 0; i < n_tensors; ++i) {
    GgufTensor t;
    uint32_t nd = 0;
    if (!r.str(&t.name) || !r.get(&nd) || nd < 1 || nd > 4)
      return fail(JEPA_E_INVALID_ARG, "gguf: tensor info %llu malformed", (unsigned long long)i);
    uint64_t n = 1;
    for (uint32_t d = 0; d < nd; ++d) {
      uint64_t e = 0;
      if (!r.get(&e) || e == 0 || e > (1ull << 40) / n)
        return fail(JEPA_E_INVALID_ARG, "gguf: tensor '%s' has an empty or oversized dimension", t.name.c_str());
      t.dims.push_back(e);
      n *= e;
    }
    if (!r.get(&t.type) || !r.get(&t.offset)) return fail(JEPA_E_INVALID_ARG, "gguf: tensor '%s' info truncated", t.name.c_str());
    const TypeInfo* ti = type_info(t.type);
    if (!ti) return fail(JEPA_E_INVALID_ARG, "gguf: tensor '%s' has unknown type %u", t.name.c_str(), t.type);
    if (t.dims[0] % ti->block)
      return fail(JEPA_E_INVALID_ARG, "gguf: tensor '%s' row of %llu is not a whole number of %s blocks", t.name.c_str(),
                  (unsigned long long)t.dims[0], ti->name);
    t.n = n;
    t.bytes = n / ti->block * ti->bytes;
    if (t.offset % g->alignment) return fail(JEPA_E_INVALID_ARG, "gguf: tensor '%s' offset not aligned", t.name.c_str());
    if (g->find(t.name)) return fail(JEPA_E_INVALID_ARG, "gguf: tensor '%s' appears twice", t.name.c_str());
    g->tensors.push_back(t);
  }
  g->data_start = (r.pos + g->alignment - 1) / g->alignment * g->alignment;
  // tensor extent: every tensor's bytes inside the file (the header alone can promise terabytes)
  for (auto& t : g->tensors) {
    if (g->data_start > r.size || t.offset > r.size - g->data_start || t.bytes > r.size - g->data_start - t.offset)
      return fail(JEPA_E_INVALID_ARG, "gguf: tensor '%s' (%llu bytes at %llu) extends past the end of the file (%llu bytes)",
                  t.name.c_str(), (unsigned long long)t.bytes, (unsigned long long)t.offset, (unsigned long long)r.size);
    t.offset += g->data_start;  // absolute from here on
  }
  return JEPA_OK;
}

const char* gguf_type_name(uint32_t type) {
  const TypeInfo* ti = type_info(type);
  return ti ? ti->name : "unknown";
}

jepa_status gguf_read_f32(const GgufFile& g, const GgufTensor& t, float* dst) {
  if (t.type != 0 && t.type != 1 && t.type != 30)
    return fail(JEPA_E_UNSUPPORTED, "gguf: tensor '%s' is %s; this build reads f32, f16 and bf16", t.name.c_str(),
                gguf_type_name(t.type));
  FILE* f = fopen(g.path.c_str(), "rb");
  if (!f) return fail(JEPA_E_INVALID_ARG, "gguf: cannot reopen '%s'", g.path.c_str());
  FileCloser closer{f};
  if (fseeko(f, (off_t)t.offset, SEEK_SET) != 0) return fail(JEPA_E_INVALID_ARG, "gguf: seek to '%s' failed", t.name.c_str());
  if (t.type == 0) {
    if (fread(dst, 4, t.n, f) != t.n) return fail(JEPA_E_INVALID_ARG, "gguf: short read of '%s'", t.name.c_str());
    return JEPA_OK;
  }
  std::vector<uint16_t> h(t.n);
  if (fread(h.data(), 2, t.n, f) != t.n) return fail(JEPA_E_INVALID_ARG, "gguf: short read of '%s'", t.name.c_str());
  if (t.type == 30) {
    for (uint64_t i = 0; i < t.n; ++i) dst[i] = jsynth_bf16_bits_to_f32(h[i]);
    return JEPA_OK;
  }
  for (uint64_t i = 0; i < t.n; ++i) {  // IEEE binary16 -> binary32, exact
    const uint32_t x = h[i], sign = (x & 0x8000u) << 16, e = (x >> 10) & 0x1f, m = x & 0x3ff;
    float v;
    if (e == 0) {
      v = std::ldexp((float)m, -24);
    } else if (e == 31) {
      v = m ? std::numeric_limits<float>::quiet_NaN() : std::numeric_limits<float>::infinity();
    } else {
      v = std::ldexp((float)(m | 0x400), (int)e - 25);
    }
    uint32_t bits;
    memcpy(&bits, &v, 4);
    bits |= sign;
    memcpy(&dst[i], &bits, 4);
  }
  return JEPA_OK;
}

}  // namespace jepa
