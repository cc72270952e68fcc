// libpkv: status strings, version, device queries and tracing shared by the entry points.
#include <cudaTypedefs.h>
#include <nvtx3/nvToolsExt.h>

#include <atomic>
#include <mutex>

#include "pkv.h"
#include "pkv_host.h"

namespace pkv {

namespace {
std::atomic<int> g_nvtx{0};  // pkv_set_nvtx
}  // namespace

NvtxRange::NvtxRange(const char* name) : on(g_nvtx.load(std::memory_order_relaxed) != 0) {
  if (on) nvtxRangePushA(name);
}
NvtxRange::~NvtxRange() {
  if (on) nvtxRangePop();
}

int device_sm_count() {
  static std::mutex mu;
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return 148;
  if (dev >= 64) dev = 63;
  std::lock_guard<std::mutex> lock(mu);
  if (cached[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
    cached[dev] = n;
  }
  return cached[dev];
}

static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static std::once_flag once;
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

namespace {

// Recently encoded tensor maps.  A serving loop calls the attention entry
// points with the same caches and shapes again and again; the encoding is pure
// host work, so its result is kept (the map holds addresses only, never data,
// and is valid on any device).  Small, most recent first, under a mutex.
struct TmapKey {
  const void* base;
  int64_t rows;
  int elt_bytes, heads, dim, box_inner, box_rows, swizzle_bytes;
  bool operator==(const TmapKey& o) const {
    return base == o.base && rows == o.rows && elt_bytes == o.elt_bytes && heads == o.heads && dim == o.dim &&
           box_inner == o.box_inner && box_rows == o.box_rows && swizzle_bytes == o.swizzle_bytes;
  }
};
constexpr int kTmapCacheSize = 16;
std::mutex g_tmap_mu;
TmapKey g_tmap_keys[kTmapCacheSize];
CUtensorMap g_tmap_maps[kTmapCacheSize];
int g_tmap_count = 0;

bool encode_tmap_3d(CUtensorMap* map, const void* base, int elt_bytes, int64_t rows, int heads, int dim,
                    int box_inner, int box_rows, int swizzle_bytes);

}  // namespace

bool make_tmap_3d(CUtensorMap* map, const void* base, int elt_bytes, int64_t rows, int heads, int dim,
                  int box_inner, int box_rows, int swizzle_bytes) {
  const TmapKey key{base, rows, elt_bytes, heads, dim, box_inner, box_rows, swizzle_bytes};
  {
    std::lock_guard<std::mutex> lock(g_tmap_mu);
    for (int i = 0; i < g_tmap_count; ++i)
      if (g_tmap_keys[i] == key) {
        *map = g_tmap_maps[i];
        return true;
      }
  }
  if (!encode_tmap_3d(map, base, elt_bytes, rows, heads, dim, box_inner, box_rows, swizzle_bytes)) return false;
  std::lock_guard<std::mutex> lock(g_tmap_mu);
  // insert at the front, dropping the oldest entry when full
  const int n = g_tmap_count < kTmapCacheSize ? g_tmap_count + 1 : kTmapCacheSize;
  for (int i = n - 1; i > 0; --i) {
    g_tmap_keys[i] = g_tmap_keys[i - 1];
    g_tmap_maps[i] = g_tmap_maps[i - 1];
  }
  g_tmap_keys[0] = key;
  g_tmap_maps[0] = *map;
  g_tmap_count = n;
  return true;
}

namespace {

bool encode_tmap_3d(CUtensorMap* map, const void* base, int elt_bytes, int64_t rows, int heads, int dim,
                    int box_inner, int box_rows, int swizzle_bytes) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t dims[3] = {(cuuint64_t)dim, (cuuint64_t)heads, (cuuint64_t)(rows > 0 ? rows : 1)};
  cuuint64_t strides[2] = {(cuuint64_t)dim * elt_bytes, (cuuint64_t)heads * dim * elt_bytes};
  cuuint32_t box[3] = {(cuuint32_t)box_inner, 1, (cuuint32_t)box_rows};
  cuuint32_t estr[3] = {1, 1, 1};
  const CUtensorMapSwizzle sw = swizzle_bytes == 128  ? CU_TENSOR_MAP_SWIZZLE_128B
                                : swizzle_bytes == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                                                      : CU_TENSOR_MAP_SWIZZLE_NONE;
  const CUtensorMapDataType dt = elt_bytes == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8;
  return fn(map, dt, 3, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace
}  // namespace pkv

extern "C" const char* pkv_status_string(int status) {
  switch (status) {
    case PKV_OK: return "PKV_OK";
    case PKV_ERR_INVALID_ARG: return "PKV_ERR_INVALID_ARG: a pointer, size or stride is invalid";
    case PKV_ERR_UNSUPPORTED: return "PKV_ERR_UNSUPPORTED: dtype, head_dim, group or block size not supported";
    case PKV_ERR_WORKSPACE: return "PKV_ERR_WORKSPACE: workspace missing or too small";
    case PKV_ERR_CUDA: return "PKV_ERR_CUDA: a CUDA launch or driver call failed";
    default: return "PKV: unknown status";
  }
}

extern "C" int pkv_abi_version(void) { return 2; }

extern "C" void pkv_set_nvtx(int on) { pkv::g_nvtx.store(on != 0 ? 1 : 0, std::memory_order_relaxed); }
