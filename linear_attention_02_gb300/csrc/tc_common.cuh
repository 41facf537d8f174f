// tc_common.cuh -- pieces shared by the tensor-core linear-attention kernels:
// chunk geometry, status bits, the phi transform of swizzled bf16 tiles,
// swizzled row stores, release/acquire flags and the TMA tensor-map encoder.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <mutex>

#include "tc_ptx.cuh"

namespace la {
namespace tcf {

using bf16 = __nv_bfloat16;
using namespace la::tc;

constexpr int L = 128;                      // chunk length = MMA M
constexpr int kThreads = 128;               // one thread per TMEM lane / tile row
constexpr uint32_t kAtom = 16384;           // one 128-row atom column (128 x 128 B)
constexpr uint32_t kWaitLimit = 1u << 24;   // mbarrier polls before giving up
constexpr uint32_t kSpinLimit = 1u << 22;   // flag polls (256 ns apart) before giving up

// Status bits written to the device error word.
constexpr unsigned kErrWait = 1u;      // a TMA or MMA completion never arrived
constexpr unsigned kErrLookback = 2u;  // an earlier span never published its state
constexpr unsigned kErrAlign = 4u;     // dynamic shared memory not 1024-byte aligned

__device__ __forceinline__ void st_release(unsigned* p, unsigned v) {
    asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ unsigned ld_acquire(const unsigned* p) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// phi on two packed bf16 values.  __expf (ex2.approx based) has a relative
// error far below the 2^-9 rounding of the bf16 result.
__device__ __forceinline__ uint32_t phi_bf16x2(uint32_t w) {
    __nv_bfloat162 h = *reinterpret_cast<__nv_bfloat162*>(&w);
    float2 f = __bfloat1622float2(h);
    f.x = f.x > 0.f ? f.x + 1.f : __expf(f.x);
    f.y = f.y > 0.f ? f.y + 1.f : __expf(f.y);
    return pack_bf16(f.x, f.y);
}

// phi in place over `atoms` swizzled atom columns; rows >= valid become 0 when
// ZERO_TAIL (padding keys must not enter S or Z: phi(0) = 1).
template <bool ZERO_TAIL>
__device__ __forceinline__ void phi_tile(uint8_t* tile, int atoms, int valid) {
    const int n = atoms * 1024;
    for (int ch = threadIdx.x; ch < n; ch += kThreads) {
        uint4* ptr = reinterpret_cast<uint4*>(tile + static_cast<size_t>(ch) * 16);
        const int row = (ch & 1023) >> 3;
        if (ZERO_TAIL && row >= valid) {
            *ptr = make_uint4(0u, 0u, 0u, 0u);
            continue;
        }
        uint4 u = *ptr;
        u.x = phi_bf16x2(u.x);
        u.y = phi_bf16x2(u.y);
        u.z = phi_bf16x2(u.z);
        u.w = phi_bf16x2(u.w);
        *ptr = u;
    }
}

// Stores 32 consecutive bf16 values (packed in pk[16]) of `row`, starting at
// column j0, into a K-major 128-row swizzled tile.
__device__ __forceinline__ void store_row32(uint8_t* tile, uint32_t atom_bytes, int row, int j0,
                                            const uint32_t (&pk)[16]) {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const int c = (j0 >> 3) + q;  // logical 16-byte chunk along the row
        *reinterpret_cast<uint4*>(tile + (c >> 3) * atom_bytes + swz(row, c & 7)) =
            make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
    }
}

// ------------------------------------------------------------------ host

using EncodeTiled = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                 const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                 const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                 CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

inline EncodeTiled encoder() {
    static EncodeTiled fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiled>(f);
    });
    return fn;
}

// 3-D map over a [BH][N][C] bf16 tensor with a {64, 128, 1} box and the
// 128-byte swizzle; rows past N read as zero and are not written.
inline cudaError_t make_map(CUtensorMap* m, const void* base, int BH, int N, int C) {
    EncodeTiled enc = encoder();
    if (!enc) return cudaErrorNotSupported;
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(C), static_cast<cuuint64_t>(N),
                          static_cast<cuuint64_t>(BH)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(C) * 2, static_cast<cuuint64_t>(N) * C * 2};
    cuuint32_t box[3] = {64, static_cast<cuuint32_t>(L), 1};
    cuuint32_t es[3] = {1, 1, 1};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides,
                     box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

}  // namespace tcf
}  // namespace la
