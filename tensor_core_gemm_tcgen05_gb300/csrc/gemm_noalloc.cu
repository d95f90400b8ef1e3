// gemm_run_noalloc: the same GEMM for callers that must not allocate device memory.
//
// gemm_create allocates the kernel's scratch (its 4-byte device error word) with
// cudaMalloc. Some callers cannot do that: code that runs where the framework owns all
// device memory and hands out none (inference-engine plugins, memory pools sized once at
// start-up), real-time loops that forbid allocation after initialisation, or library code
// that must not touch the allocator at all. This entry point needs no context: the
// kernel's scratch lives in a file-scope __device__ array that every GPU loading this
// library holds until the process exits.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>
#include <functional>
#include <mutex>

#include "gemm.h"
#include "gemm_kernel.cuh"
#include "softmax_gemm_kernel.cuh"

// The scratch of gemm_run_noalloc, GEMM_NOALLOC_SCRATCH_BYTES (256) bytes on every device.
// Word 0 is the kernel's error word (which in-kernel wait ran out, 0 if none). In host code
// this name is only a host-side stand-in: its device address comes from
// cudaGetSymbolAddress, taken once per device during set-up.
static __device__ __align__(256) uint32_t g_noalloc_scratch[GEMM_NOALLOC_SCRATCH_BYTES / sizeof(uint32_t)];

namespace {

// Same tile configuration as gemm_run's kernel, as a type of its own, so that this file's
// kernel instance (and its shared-memory attribute) is separate from the one in gemm_api.cu.
struct NoAllocCfg : gb300::KernelConfig<128, 256, 4> {};
// The softmax epilogue's kernel (one CTA per 128-row block, N <= 256), likewise its own type.
struct NoAllocSoftCfg : gb300::SoftmaxConfig<3> {};
constexpr int kGroupM = 16;
constexpr uint64_t kTimeoutNs = 2000000000ull;
constexpr int kMaxDevices = 64;
// Scratch this kernel needs for any problem size: one 32-bit error word.
constexpr size_t kScratchNeed = sizeof(uint32_t);
static_assert(kScratchNeed <= GEMM_NOALLOC_SCRATCH_BYTES, "scratch array too small");

struct DeviceSetup {
    std::once_flag once;
    int status = GEMM_ERR_DEVICE;
    int num_sms = 0;
    PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
    uint32_t *scratch = nullptr;   // device address of g_noalloc_scratch on this device
};

DeviceSetup g_setup[kMaxDevices];

// Runs once per device, with that device current.
void setup_device(DeviceSetup &s, int device)
{
    int major = 0, minor = 0, sms = 0, smem_optin = 0;
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, device);
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, device);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device);
    cudaDeviceGetAttribute(&smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, device);
    if (major != 10 || minor != 3 || sms <= 0 || smem_optin < NoAllocCfg::SMEM_BYTES ||
        smem_optin < NoAllocSoftCfg::SMEM_BYTES) {
        cudaGetLastError();
        s.status = GEMM_ERR_DEVICE;
        return;
    }
    if (cudaFuncSetAttribute(gb300::gemm_tcgen05_kernel<NoAllocCfg>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             NoAllocCfg::SMEM_BYTES) != cudaSuccess ||
        cudaFuncSetAttribute(gb300::gemm_softmax_kernel<NoAllocSoftCfg, false>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, NoAllocSoftCfg::SMEM_BYTES) != cudaSuccess) {
        cudaGetLastError();
        s.status = GEMM_ERR_DEVICE;
        return;
    }
    void *fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !fn) {
        cudaGetLastError();
        s.status = GEMM_ERR_DEVICE;
        return;
    }
    void *ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || !ptr) {
        cudaGetLastError();
        s.status = GEMM_ERR_LAUNCH;
        return;
    }
    s.encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    s.scratch = static_cast<uint32_t *>(ptr);
    s.num_sms = sms;
    s.status = GEMM_OK;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool on_device(const void *p, int device)
{
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    return a.type == cudaMemoryTypeManaged || (a.type == cudaMemoryTypeDevice && a.device == device);
}

bool overlaps(const void *a, size_t na, const void *b, size_t nb)
{
    if (!a || !b || na == 0 || nb == 0)
        return false;
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
    return a0 < b0 + nb && b0 < a0 + na;
}

bool encode_2d(PFN_cuTensorMapEncodeTiled_v12000 encode, CUtensorMap *map, const void *ptr, uint64_t inner,
               uint64_t outer, uint32_t box_inner, uint32_t box_outer,
               CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B)
{
    const cuuint64_t dims[2] = {inner, outer};
    const cuuint64_t strides[1] = {inner * 2};
    const cuuint32_t box[2] = {box_inner, box_outer};
    const cuuint32_t estr[2] = {1, 1};
    return encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void *>(ptr), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

extern "C" int gemm_run_noalloc(int64_t M, int64_t N, int64_t K, const void *A, const void *B, const void *bias,
                                void *C, int epilogue, void *stream)
{
    // Largest problem: M, N, K <= 2^31 - 1 (32-bit TMA coordinates); the scratch it needs
    // (kScratchNeed) is the same for every size and fits the array.
    if (M < 0 || N < 0 || K < 0 || M > INT32_MAX || N > INT32_MAX || K > INT32_MAX)
        return GEMM_ERR_ARG;
    if (epilogue < GEMM_EPI_NONE || epilogue > GEMM_EPI_SOFTMAX)
        return GEMM_ERR_ARG;
    if (epilogue == GEMM_EPI_SOFTMAX && N > 256)
        return GEMM_ERR_ARG;   // the fused softmax needs whole rows inside one tile
    if (M == 0 || N == 0)
        return GEMM_OK;
    if (!C || (K > 0 && (!A || !B)))
        return GEMM_ERR_ARG;
    if (N % 8 != 0 || K % 8 != 0)
        return GEMM_ERR_ALIGN;
    if (!aligned16(C) || (K > 0 && (!aligned16(A) || !aligned16(B))) || (bias && !aligned16(bias)))
        return GEMM_ERR_ALIGN;
    const size_t cb = static_cast<size_t>(M) * N * 2;
    if (overlaps(C, cb, A, static_cast<size_t>(M) * K * 2) || overlaps(C, cb, B, static_cast<size_t>(K) * N * 2) ||
        overlaps(C, cb, bias, static_cast<size_t>(N) * 2))
        return GEMM_ERR_ARG;

    int device = -1;
    if (cudaGetDevice(&device) != cudaSuccess || device < 0 || device >= kMaxDevices) {
        cudaGetLastError();
        return GEMM_ERR_DEVICE;
    }
    DeviceSetup &s = g_setup[device];
    std::call_once(s.once, setup_device, std::ref(s), device);
    if (s.status != GEMM_OK)
        return s.status;
    if (!on_device(C, device) || (K > 0 && (!on_device(A, device) || !on_device(B, device))) ||
        (bias && !on_device(bias, device)))
        return GEMM_ERR_DEVICE;

    CUtensorMap ta, tb, tc;
    std::memset(&ta, 0, sizeof(ta));
    std::memset(&tb, 0, sizeof(tb));
    if (K > 0) {
        if (!encode_2d(s.encode, &ta, A, static_cast<uint64_t>(K), static_cast<uint64_t>(M), NoAllocCfg::BK,
                       NoAllocCfg::BM) ||
            !encode_2d(s.encode, &tb, B, static_cast<uint64_t>(N), static_cast<uint64_t>(K), NoAllocCfg::B_BOX_N,
                       NoAllocCfg::BK))
            return GEMM_ERR_LAUNCH;
    }
    // the GEMM kernel stores 32 x 32 boxes (64-byte swizzle), the softmax kernel 32-row x
    // 64-column boxes (128-byte swizzle)
    const bool smx = epilogue == GEMM_EPI_SOFTMAX;
    if (!encode_2d(s.encode, &tc, C, static_cast<uint64_t>(N), static_cast<uint64_t>(M), smx ? 64 : 32, 32,
                   smx ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B))
        return GEMM_ERR_LAUNCH;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    // The array keeps the previous call's contents: the error word must start at zero.
    if (cudaMemsetAsync(s.scratch, 0, kScratchNeed, st) != cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_LAUNCH;
    }
    gb300::GemmParams p;
    p.M = static_cast<int>(M);
    p.N = static_cast<int>(N);
    p.K = static_cast<int>(K);
    p.m_blocks = (p.M + NoAllocCfg::BM - 1) / NoAllocCfg::BM;
    p.n_blocks = (p.N + NoAllocCfg::BN - 1) / NoAllocCfg::BN;
    p.num_tiles = p.m_blocks * p.n_blocks;
    p.num_kb = (p.K + NoAllocCfg::BK - 1) / NoAllocCfg::BK;
    p.group_m = kGroupM;   // row blocks per raster group
    p.epilogue = epilogue;
    p.bias = static_cast<const __half *>(bias);
    p.C = static_cast<__half *>(C);
    p.ldc = N;   // C is tightly packed
    p.err = s.scratch;
    p.timeout_ns = kTimeoutNs;
    p.debug = 0;
    const int grid = p.num_tiles < s.num_sms ? p.num_tiles : s.num_sms;
    if (epilogue == GEMM_EPI_SOFTMAX) {
        // the row fits one tile: one CTA per 128-row block (a cluster of one), a single pass
        p.row_cluster = 1;
        p.smx_span = 1;
        p.smx_two_pass = 0;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
        cfg.blockDim = dim3(NoAllocSoftCfg::NUM_THREADS, 1, 1);
        cfg.dynamicSmemBytes = NoAllocSoftCfg::SMEM_BYTES;
        cfg.stream = st;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 1;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        cudaLaunchKernelEx(&cfg, gb300::gemm_softmax_kernel<NoAllocSoftCfg, false>, ta, tb, tc, p);
    } else {
        gb300::gemm_tcgen05_kernel<NoAllocCfg><<<grid, NoAllocCfg::NUM_THREADS, NoAllocCfg::SMEM_BYTES, st>>>(ta, tb, tc,
                                                                                                          p);
    }
    if (cudaGetLastError() != cudaSuccess)
        return GEMM_ERR_LAUNCH;
    return GEMM_OK;
}
