// Host side of the TMA staging: tensor maps encoded with cuTensorMapEncodeTiled,
// reached through the runtime's driver entry point (no link against libcuda).
//
// A tensor map is a pure function of its parameters (data type, rank, global
// address, extents, strides, box, swizzle), and a layer's calls reuse the
// same buffers, so encoded maps are kept in a small hash table keyed by all of
// them: a bf16 forward then costs lookups instead of a dozen driver calls.
#include <cstring>
#include <mutex>

#include "ptx.cuh"

namespace moe {
namespace {

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  // looked up once per process (a thread-safe function-local initialisation)
  static const EncodeTiledFn fn = []() -> EncodeTiledFn {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      return (EncodeTiledFn)p;
    return nullptr;
  }();
  return fn;
}

// Every parameter of an encoding (the ones fixed here -- unit element
// strides, no interleave, 256-byte L2 promotion, zero fill -- are the same for
// every map of this library).
struct MapKey {
  uint32_t dtype, rank, swizzle, pad;
  uint64_t ptr;
  uint64_t dims[3], strides[2];
  uint32_t box[3], pad2;
};
struct MapSlot {
  bool used;
  MapKey key;
  CUtensorMap map;
};
constexpr int kMapSlots = 256;
std::mutex g_map_mutex;
MapSlot g_maps[kMapSlots];

bool encode(CUtensorMap* m, CUtensorMapDataType dtype, uint32_t rank, const void* ptr, const cuuint64_t* dims,
            const cuuint64_t* strides, const cuuint32_t* box, CUtensorMapSwizzle sw) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  MapKey k;
  memset(&k, 0, sizeof(k));
  k.dtype = (uint32_t)dtype;
  k.rank = rank;
  k.swizzle = (uint32_t)sw;
  k.ptr = (uint64_t)(uintptr_t)ptr;
  for (uint32_t i = 0; i < rank; ++i) {
    k.dims[i] = dims[i];
    k.box[i] = box[i];
    if (i + 1 < rank) k.strides[i] = strides[i];
  }
  // FNV-1a over the key's bytes picks the slot; a collision re-encodes.
  uint64_t h = 1469598103934665603ull;
  const unsigned char* b = reinterpret_cast<const unsigned char*>(&k);
  for (size_t i = 0; i < sizeof(k); ++i) h = (h ^ b[i]) * 1099511628211ull;
  MapSlot& slot = g_maps[h % kMapSlots];
  std::lock_guard<std::mutex> lock(g_map_mutex);
  if (slot.used && memcmp(&slot.key, &k, sizeof(k)) == 0) {
    *m = slot.map;
    return true;
  }
  const cuuint32_t es[3] = {1, 1, 1};
  if (enc(m, dtype, rank, const_cast<void*>(ptr), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return false;
  slot.used = true;
  slot.key = k;
  slot.map = *m;
  return true;
}

}  // namespace

bool tmap_bf16_2d(CUtensorMap* m, const void* ptr, int64_t rows, int64_t cols, int box_cols, int box_rows) {
  return tmap_bf16_2d_swizzle(m, ptr, rows, cols, box_cols, box_rows, 128);
}

bool tmap_bf16_2d_swizzle(CUtensorMap* m, const void* ptr, int64_t rows, int64_t cols, int box_cols, int box_rows,
                          int row_bytes) {
  if (rows <= 0 || cols <= 0) return false;
  CUtensorMapSwizzle sw;
  switch (row_bytes) {
    case 16: sw = CU_TENSOR_MAP_SWIZZLE_NONE; break;
    case 32: sw = CU_TENSOR_MAP_SWIZZLE_32B; break;
    case 64: sw = CU_TENSOR_MAP_SWIZZLE_64B; break;
    case 128: sw = CU_TENSOR_MAP_SWIZZLE_128B; break;
    default: return false;
  }
  if (box_cols * 2 != row_bytes) return false;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
  cuuint32_t box[2] = {(cuuint32_t)box_cols, (cuuint32_t)box_rows};
  return encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, ptr, dims, strides, box, sw);
}

bool tmap_bf16_3d(CUtensorMap* m, const void* ptr, int G, int64_t rows, int64_t cols, int box_cols, int box_rows) {
  if (G <= 0 || rows <= 0 || cols <= 0) return false;
  cuuint64_t dims[3] = {(cuuint64_t)cols, (cuuint64_t)rows, (cuuint64_t)G};
  cuuint64_t strides[2] = {(cuuint64_t)cols * 2, (cuuint64_t)rows * cols * 2};
  cuuint32_t box[3] = {(cuuint32_t)box_cols, (cuuint32_t)box_rows, 1};
  return encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, ptr, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
}

bool tmap_f32_2d(CUtensorMap* m, const void* ptr, int64_t rows, int64_t cols, int box_rows) {
  if (rows <= 0 || cols <= 0 || cols % 4 != 0) return false;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)cols * 4};
  cuuint32_t box[2] = {32u, (cuuint32_t)box_rows};
  return encode(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, ptr, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
}

bool tmap_u8_2d(CUtensorMap* m, const void* ptr, int64_t rows, int64_t cols, int box_rows) {
  if (rows <= 0 || cols <= 0 || cols % 16 != 0) return false;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)cols};
  cuuint32_t box[2] = {128u, (cuuint32_t)box_rows};
  return encode(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, ptr, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
}

bool tmap_u8_3d(CUtensorMap* m, const void* ptr, int G, int64_t rows, int64_t cols, int box_rows) {
  if (G <= 0 || rows <= 0 || cols <= 0 || cols % 16 != 0) return false;
  cuuint64_t dims[3] = {(cuuint64_t)cols, (cuuint64_t)rows, (cuuint64_t)G};
  cuuint64_t strides[2] = {(cuuint64_t)cols, (cuuint64_t)rows * cols};
  cuuint32_t box[3] = {128u, (cuuint32_t)box_rows, 1};
  return encode(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, ptr, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
}

}  // namespace moe
