// Host helpers for the TMA tensor maps of the tcgen05 kernels (router_gemm.cu,
// expert_mlp.cu): BF16 row-major matrices (boxes of 64 columns) and FP8 byte matrices
// (boxes of 128 columns), both with the 128-byte swizzle. Encoded maps are kept in a small
// per-thread cache keyed by the encoder's arguments.
#include <mutex>

#include "internal.cuh"

namespace beam {
namespace {

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// The driver's encoder, fetched through the runtime once (the library does not link libcuda).
EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// Encoded maps of this thread's recent calls, keyed by every encoder argument. A map is a
// pure function of those arguments, so a hit is exactly what a new encoding would give;
// steady-state calls (same weights, same pool scratch addresses) encode nothing.
struct CachedMap {
    bool used = false;
    CUtensorMapDataType dtype;
    const void* base;
    uint64_t rows, cols, row_bytes;
    uint32_t box_rows, box_cols;
    CUtensorMapSwizzle swizzle;
    CUtensorMap map;
};
constexpr int kCacheEntries = 64;
thread_local CachedMap g_cache[kCacheEntries];
thread_local int g_cache_next = 0;

bool encode_2d(CUtensorMap* map, CUtensorMapDataType dtype, const void* base, uint64_t rows, uint64_t cols,
               uint64_t row_bytes, uint32_t box_rows, uint32_t box_cols, const char** why,
               CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B) {
    for (const CachedMap& c : g_cache) {
        if (c.used && c.dtype == dtype && c.base == base && c.rows == rows && c.cols == cols &&
            c.row_bytes == row_bytes && c.box_rows == box_rows && c.box_cols == box_cols && c.swizzle == swizzle) {
            *map = c.map;
            return true;
        }
    }
    EncodeTiledFn fn = encode_fn();
    if (!fn) {
        *why = "driver entry point cuTensorMapEncodeTiled is not available";
        return false;
    }
    const cuuint64_t dims[2] = {cols, rows};
    const cuuint64_t strides[1] = {row_bytes};
    const cuuint32_t box[2] = {box_cols, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = fn(map, dtype, 2, const_cast<void*>(base), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        *why = "cuTensorMapEncodeTiled rejected a tensor map";
        return false;
    }
    CachedMap& c = g_cache[g_cache_next];
    g_cache_next = (g_cache_next + 1) % kCacheEntries;
    c.used = true;
    c.dtype = dtype;
    c.base = base;
    c.rows = rows;
    c.cols = cols;
    c.row_bytes = row_bytes;
    c.box_rows = box_rows;
    c.box_cols = box_cols;
    c.swizzle = swizzle;
    c.map = *map;
    return true;
}

}  // namespace

bool encode_tmap_bf16_2d(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows,
                         uint32_t box_cols, const char** why) {
    return encode_2d(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, base, rows, cols, cols * 2, box_rows, box_cols, why);
}

bool encode_tmap_u8_2d(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows,
                       uint32_t box_cols, const char** why) {
    return encode_2d(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, base, rows, cols, cols, box_rows, box_cols, why);
}

bool encode_bmaps(BMaps* b, const void* base, uint64_t rows, uint64_t cols, int bn_max, const char** why) {
    for (int i = 0; i < kBoxKinds; ++i) {
        const uint32_t h = kBoxRows << i;
        if (static_cast<int>(h) > bn_max) {
            b->m[i] = b->m[0];
            continue;
        }
        if (!encode_tmap_bf16_2d(&b->m[i], base, rows, cols, h, kTileK, why)) return false;
    }
    return true;
}

bool encode_tmap_u8_2d_plain(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows,
                             uint32_t box_cols, const char** why) {
    return encode_2d(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, base, rows, cols, cols, box_rows, box_cols, why,
                     CU_TENSOR_MAP_SWIZZLE_NONE);
}

bool encode_bmaps_u8(BMaps* b, const void* base, uint64_t rows, uint64_t cols, int box_max, const char** why) {
    for (int i = 0; i < kBoxKinds; ++i) {
        const uint32_t h = kBoxRows << i;
        if (static_cast<int>(h) > box_max) {
            b->m[i] = b->m[0];
            continue;
        }
        if (!encode_tmap_u8_2d(&b->m[i], base, rows, cols, h, 128, why)) return false;
    }
    return true;
}

}  // namespace beam
