// Host-side helpers: device capability cache, tensor-map encoding, status names.
#include <mutex>

#include "common.cuh"

namespace dflash2 {

namespace {
constexpr int kMaxDevices = 64;
DeviceInfo g_info[kMaxDevices];
bool g_have[kMaxDevices];
std::mutex g_mu;

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                   const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                   const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;
}  // namespace

dflash2_status current_device(DeviceInfo *info) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return DFLASH2_ERR_CUDA;
    }
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_have[dev]) {
        DeviceInfo d{};
        d.device = dev;
        int major = 0, minor = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&d.max_smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) !=
                cudaSuccess) {
            cudaGetLastError();
            return DFLASH2_ERR_CUDA;
        }
        d.supported = (major == 10 && minor == 3);
        g_info[dev] = d;
        g_have[dev] = true;
    }
    *info = g_info[dev];
    return g_info[dev].supported ? DFLASH2_OK : DFLASH2_ERR_UNSUPPORTED_DEVICE;
}

dflash2_status encode_tmap_bf16(CUtensorMap *map, const void *base, uint64_t rows, uint64_t cols,
                                uint32_t box_rows) {
    return encode_tmap_2d(map, base, rows, cols, box_rows, 2);
}

// Resolves cuTensorMapEncodeTiled once (through the runtime, so the
// library needs no link against libcuda).
static dflash2_status resolve_encode() {
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_encode) {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                             cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess || !fn) {
            cudaGetLastError();
            return DFLASH2_ERR_CUDA;
        }
        g_encode = reinterpret_cast<EncodeTiledFn>(fn);
    }
    return DFLASH2_OK;
}

dflash2_status encode_tmap_2d(CUtensorMap *map, const void *base, uint64_t rows, uint64_t cols,
                              uint32_t box_rows, uint32_t elem_bytes) {
    const dflash2_status st = resolve_encode();
    if (st != DFLASH2_OK) return st;
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {cols * elem_bytes};
    cuuint32_t box[2] = {128 / elem_bytes, box_rows};  // one 128-byte swizzle row wide
    cuuint32_t estr[2] = {1, 1};
    const CUtensorMapDataType type =
        elem_bytes == 1 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    CUresult r = g_encode(map, type, 2, const_cast<void *>(base), dims,
                          strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? DFLASH2_OK : DFLASH2_ERR_CUDA;
}

// Plain (unswizzled) byte rows: box of box_cols bytes (<= 256, a multiple
// of 16) x box_rows rows.
dflash2_status encode_tmap_bytes_2d(CUtensorMap *map, const void *base, uint64_t rows,
                                    uint64_t cols, uint32_t box_cols, uint32_t box_rows) {
    const dflash2_status st = resolve_encode();
    if (st != DFLASH2_OK) return st;
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {cols};
    cuuint32_t box[2] = {box_cols, box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(base), dims,
                          strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? DFLASH2_OK : DFLASH2_ERR_CUDA;
}

}  // namespace dflash2

extern "C" const char *dflash2_status_string(int32_t status) {
    switch (status) {
        case DFLASH2_OK: return "ok";
        case DFLASH2_ERR_INVALID_ARG: return "invalid argument";
        case DFLASH2_ERR_UNSUPPORTED_DTYPE: return "unsupported dtype (fp32 or bf16 only)";
        case DFLASH2_ERR_MISALIGNED: return "misaligned pointer or stride";
        case DFLASH2_ERR_WORKSPACE: return "workspace missing or too small";
        case DFLASH2_ERR_CUDA: return "CUDA runtime error";
        case DFLASH2_ERR_UNSUPPORTED_DEVICE: return "device is not sm_103 (GB300)";
        default: return "unknown status";
    }
}

extern "C" int32_t dflash2_abi_version(void) { return DFLASH2_ABI_VERSION; }
