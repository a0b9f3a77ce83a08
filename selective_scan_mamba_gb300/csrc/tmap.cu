// tmap.cu -- host-side encoding of TMA tensor maps.  The driver entry point
// cuTensorMapEncodeTiled is fetched through the runtime, so the library needs no
// link-time dependency on libcuda.  A map is a pure function of its arguments (address,
// element type, shape, box, swizzle), so the last kMapCache encodings are kept and a
// repeated call (a training or decode loop over the same buffers) copies the cached map
// instead of encoding it again.  The shared-memory attribute of a kernel is likewise set
// once per (device, kernel, size).
#include <cuda.h>
#include <cuda_runtime.h>
#include <cstring>
#include <mutex>

#include "launch.h"

namespace ssm {

namespace {

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

std::mutex g_mu;
EncodeTiledFn g_encode = nullptr;

struct MapKey {
    const void* base;
    int kind, elem_bytes, rank, swizzle;  // kind: 2-D or n-D encoder
    unsigned long long dims[5];
    unsigned box[5];
    bool operator==(const MapKey& o) const { return std::memcmp(this, &o, sizeof(MapKey)) == 0; }
};
constexpr int kMapCache = 64;
struct MapEntry {
    MapKey key;
    CUtensorMap map;
    unsigned long long used;  // 0: empty
};
MapEntry g_maps[kMapCache];
unsigned long long g_tick = 0;

MapKey make_key(int kind, const void* base, int elem_bytes, int rank, const unsigned long long* dims,
                const unsigned* box, bool swizzle128) {
    MapKey k;
    std::memset(&k, 0, sizeof(k));  // padding too: keys compare as bytes
    k.kind = kind;
    k.base = base;
    k.elem_bytes = elem_bytes;
    k.rank = rank;
    k.swizzle = swizzle128 ? 1 : 0;
    for (int i = 0; i < rank && i < 5; ++i) {
        k.dims[i] = dims[i];
        k.box[i] = box[i];
    }
    return k;
}

bool cached_map(const MapKey& k, CUtensorMap* out) {
    std::lock_guard<std::mutex> lock(g_mu);
    for (MapEntry& e : g_maps) {
        if (e.used != 0 && e.key == k) {
            e.used = ++g_tick;
            *out = e.map;
            return true;
        }
    }
    return false;
}

void keep_map(const MapKey& k, const CUtensorMap& m) {
    std::lock_guard<std::mutex> lock(g_mu);
    MapEntry* victim = &g_maps[0];
    for (MapEntry& e : g_maps) {
        if (e.used < victim->used) victim = &e;
    }
    victim->key = k;
    victim->map = m;
    victim->used = ++g_tick;
}

cudaError_t encoder(EncodeTiledFn* out) {
    std::lock_guard<std::mutex> lock(g_mu);
    if (g_encode == nullptr) {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                         cudaEnableDefault, &q);
        if (e != cudaSuccess) return e;
        if (q != cudaDriverEntryPointSuccess || fn == nullptr) return cudaErrorNotSupported;
        g_encode = reinterpret_cast<EncodeTiledFn>(fn);
    }
    *out = g_encode;
    return cudaSuccess;
}

}  // namespace

// 2-D row-major tensor [rows][inner] of 2- or 4-byte elements, 128-byte swizzled boxes of
// box_inner x box_rows elements, zero fill outside the tensor.
cudaError_t encode_tmap_2d(CUtensorMap* map, const void* base, int elem_bytes,
                           unsigned long long inner, unsigned long long rows, unsigned box_inner,
                           unsigned box_rows, bool swizzle128) {
    const unsigned long long kd[2] = {inner, rows};
    const unsigned kb[2] = {box_inner, box_rows};
    const MapKey key = make_key(2, base, elem_bytes, 2, kd, kb, swizzle128);
    if (cached_map(key, map)) return cudaSuccess;
    EncodeTiledFn fn = nullptr;
    cudaError_t e = encoder(&fn);
    if (e != cudaSuccess) return e;
    const CUtensorMapDataType dt =
        elem_bytes == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
    const cuuint64_t dims[2] = {inner, rows};
    const cuuint64_t strides[1] = {inner * static_cast<uint64_t>(elem_bytes)};
    const cuuint32_t box[2] = {box_inner, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(map, dt, 2, const_cast<void*>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE,
                    swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
    keep_map(key, *map);
    return cudaSuccess;
}

// Row-major tensor of `rank` dimensions (dims[0] innermost), contiguous strides.
cudaError_t encode_tmap_nd(CUtensorMap* map, const void* base, int elem_bytes, int rank,
                           const unsigned long long* dims, const unsigned* box, bool swizzle128) {
    if (rank < 1 || rank > 5) return cudaErrorInvalidValue;
    const MapKey key = make_key(0, base, elem_bytes, rank, dims, box, swizzle128);
    if (cached_map(key, map)) return cudaSuccess;
    EncodeTiledFn fn = nullptr;
    cudaError_t e = encoder(&fn);
    if (e != cudaSuccess) return e;
    const CUtensorMapDataType dt =
        elem_bytes == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
    cuuint64_t gd[5], gs[4];
    cuuint32_t bx[5], es[5];
    unsigned long long stride = static_cast<unsigned long long>(elem_bytes);
    for (int i = 0; i < rank; ++i) {
        gd[i] = dims[i];
        bx[i] = box[i];
        es[i] = 1;
        if (i > 0) gs[i - 1] = stride;
        stride *= dims[i];
    }
    CUresult r = fn(map, dt, static_cast<cuuint32_t>(rank), const_cast<void*>(base), gd, gs, bx, es,
                    CU_TENSOR_MAP_INTERLEAVE_NONE,
                    swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
    keep_map(key, *map);
    return cudaSuccess;
}

// cudaFuncSetAttribute(MaxDynamicSharedMemorySize) only when a launch needs more than the
// kernel's limit already set on this device: the attribute is an upper bound, so the
// largest value set so far serves every smaller launch.  The last kAttrCache (device,
// kernel) pairs are remembered.
cudaError_t set_smem_attr(const void* kernel, int bytes) {
    constexpr int kAttrCache = 256;
    struct Entry {
        const void* fn;
        int dev, bytes;
    };
    static Entry seen[kAttrCache];
    static int next = 0;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    {
        std::lock_guard<std::mutex> lock(g_mu);
        for (const Entry& s : seen)
            if (s.fn == kernel && s.dev == dev && s.bytes >= bytes) return cudaSuccess;
    }
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lock(g_mu);
    for (Entry& s : seen) {
        if (s.fn == kernel && s.dev == dev) {  // raise the remembered limit
            if (bytes > s.bytes) s.bytes = bytes;
            return cudaSuccess;
        }
    }
    seen[next] = Entry{kernel, dev, bytes};
    next = (next + 1) % kAttrCache;
    return cudaSuccess;
}

}  // namespace ssm
