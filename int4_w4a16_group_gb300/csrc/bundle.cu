// Multi-tensor weight bundle: one file holding the packed codes (.qw) and group scales (.sc) of
// many named linears, loaded into a caller-provided device arena and registered by name for
// linear() dispatch.
//
// Page "The Final Wire: How a Single Edit Integrated INT4 Quantization into a Native DDTree
// Inference Engine", section "The Multi-Step Integration Chain", steps 3 and 5: a generator
// writes bundles of quantized weights and scales, and the engine keeps maps from weight names to
// them. The pages do not give the bundle's byte layout; this one is the library's own:
//
//   offset 0   8 bytes  magic "W4A16BDL"
//              u32      version (1)
//              u32      count
//   entries    count x { u32 name_len; name bytes (no terminator); i32 K; i32 N;
//                        u64 qw_offset; u64 sc_offset }
//   data       the blobs at their offsets: qw [K/8, N] int32, sc [K/32, N] float32, row-major
//
// All integers little-endian. The loader checks every field against the file size before it
// copies anything.
#include <cuda_runtime.h>
#include <stdio.h>
#include <string.h>

#include <set>
#include <string>
#include <vector>

#include "../../include/w4a16.h"
#include "internal.h"

namespace {

struct BundleEntry {
  std::string name;
  int K, N;
  uint64_t qoff, soff, qbytes, sbytes;
};

constexpr uint32_t kMaxEntries = 1u << 20;
constexpr uint32_t kMaxName = 4096;

size_t align256(size_t v) { return (v + 255) & ~(size_t)255; }

struct File {
  FILE* f = nullptr;
  ~File() {
    if (f) fclose(f);
  }
};

bool read_exact(FILE* f, void* dst, size_t n) { return fread(dst, 1, n, f) == n; }

// Reads and checks the index; W4A16_ERR_IO for unreadable or malformed files.
w4a16_status parse(const char* path, std::vector<BundleEntry>& out) {
  File file;
  file.f = fopen(path, "rb");
  if (!file.f) return W4A16_ERR_IO;
  if (fseeko(file.f, 0, SEEK_END) != 0) return W4A16_ERR_IO;
  const long long fsize_s = (long long)ftello(file.f);
  if (fsize_s < 16 || fseeko(file.f, 0, SEEK_SET) != 0) return W4A16_ERR_IO;
  const uint64_t fsize = (uint64_t)fsize_s;
  char magic[8];
  uint32_t version = 0, count = 0;
  if (!read_exact(file.f, magic, 8) || memcmp(magic, "W4A16BDL", 8) != 0) return W4A16_ERR_IO;
  if (!read_exact(file.f, &version, 4) || !read_exact(file.f, &count, 4)) return W4A16_ERR_IO;
  if (version != 1 || count > kMaxEntries) return W4A16_ERR_IO;
  std::set<std::string> names;
  out.clear();
  for (uint32_t i = 0; i < count; ++i) {
    uint32_t len = 0;
    if (!read_exact(file.f, &len, 4) || len == 0 || len > kMaxName) return W4A16_ERR_IO;
    std::string name(len, '\0');
    if (!read_exact(file.f, &name[0], len)) return W4A16_ERR_IO;
    if (name.find('\0') != std::string::npos || !names.insert(name).second) return W4A16_ERR_IO;
    BundleEntry e;
    e.name = name;
    if (!read_exact(file.f, &e.K, 4) || !read_exact(file.f, &e.N, 4) ||
        !read_exact(file.f, &e.qoff, 8) || !read_exact(file.f, &e.soff, 8))
      return W4A16_ERR_IO;
    if (e.K <= 0 || e.K % W4A16_GROUP != 0 || e.N <= 0 || e.N % 4 != 0) return W4A16_ERR_IO;
    e.qbytes = (uint64_t)(e.K / 8) * (uint64_t)e.N * 4u;
    e.sbytes = (uint64_t)(e.K / W4A16_GROUP) * (uint64_t)e.N * 4u;
    if (e.qoff > fsize || e.qbytes > fsize - e.qoff || e.soff > fsize ||
        e.sbytes > fsize - e.soff)
      return W4A16_ERR_IO;
    out.push_back(e);
  }
  return W4A16_OK;
}

size_t arena_bytes(const std::vector<BundleEntry>& v) {
  size_t total = 0;
  for (const auto& e : v) total += align256(e.qbytes) + align256(e.sbytes);
  return total;
}

}  // namespace

extern "C" {

w4a16_status w4a16_bundle_info(const char* path, int* count, size_t* device_bytes) {
  if (!path) return W4A16_ERR_ARG;
  std::vector<BundleEntry> v;
  const w4a16_status st = parse(path, v);
  if (st != W4A16_OK) return st;
  if (count) *count = (int)v.size();
  if (device_bytes) *device_bytes = arena_bytes(v);
  return W4A16_OK;
}

w4a16_status w4a16_bundle_load(w4a16_registry* reg, const char* path, void* arena,
                               size_t arena_size) {
  if (!reg || !path) return W4A16_ERR_ARG;
  std::vector<BundleEntry> v;
  w4a16_status st = parse(path, v);
  if (st != W4A16_OK) return st;
  const size_t need = arena_bytes(v);
  if (need > 0 && (!arena || arena_size < need)) return W4A16_ERR_WORKSPACE;
  if (((uintptr_t)arena & 255u) != 0) return W4A16_ERR_ALIGN;
  File file;
  file.f = fopen(path, "rb");
  if (!file.f) return W4A16_ERR_IO;
  std::vector<char> buf;
  char* dst = static_cast<char*>(arena);
  for (const auto& e : v) {
    char* qd = dst;
    char* sd = dst + align256(e.qbytes);
    dst = sd + align256(e.sbytes);
    const uint64_t offs[2] = {e.qoff, e.soff};
    const uint64_t sizes[2] = {e.qbytes, e.sbytes};
    char* dsts[2] = {qd, sd};
    for (int k = 0; k < 2; ++k) {
      buf.resize(sizes[k]);
      if (fseeko(file.f, (off_t)offs[k], SEEK_SET) != 0 ||
          !read_exact(file.f, buf.data(), sizes[k]))
        return W4A16_ERR_IO;
      const cudaError_t ce = cudaMemcpy(dsts[k], buf.data(), sizes[k], cudaMemcpyHostToDevice);
      if (ce != cudaSuccess) return W4A16_ERR_CUDA;
    }
    st = w4a16_registry_add(reg, e.name.c_str(), reinterpret_cast<const int32_t*>(qd),
                            reinterpret_cast<const float*>(sd), e.K, e.N, W4A16_GROUP);
    if (st != W4A16_OK) return st;
  }
  return W4A16_OK;
}

}  // extern "C"
