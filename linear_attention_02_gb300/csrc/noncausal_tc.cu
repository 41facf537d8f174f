// noncausal_tc.cu -- non-causal linear attention for fp32 storage on the
// 5th-generation tensor core, D = M = 64.
//
// V' = phi(Q) (phi(K)^T V) / phi(Q) sum_j phi(K_j)  ("Transformers are RNNs",
// section 二, eq. linear): every query reads the same state S = phi(K)^T V and
// Z = sum phi(K), so the work is two passes -- build the state, then read it.
//
// fp32 operands run on the bf16 tensor path split in two: x = hi + lo with
// hi = bf16(x) and lo = bf16(x - hi), and a product a b is taken as
// a_hi b_hi + a_hi b_lo + a_lo b_hi (the dropped a_lo b_lo and the rounding of
// the lo parts are about 2^-17 of |a b|), accumulated in fp32 in TMEM.  The
// ones block appended to V carries the normaliser through the same products.
//
//   state kernel   one CTA per (head, span): TMA loads fp32 K, V tiles of 128
//                  tokens; phi and the split are done in place (the fp32 tile
//                  becomes its hi and lo bf16 tiles); the MMAs accumulate
//                  [S | Z] for the span, published as fp32 partials;
//   read-out kernel one CTA per (head, span): sums the partials of the head,
//                  splits [S | Z] into bf16 hi and lo state tiles, then per
//                  chunk loads fp32 Q, applies phi and the split, takes the
//                  three products into TMEM and stores num / den as fp32.
// Each input is read once from HBM and the output written once.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>

#include "la_launch.h"
#include "tc_common.cuh"

namespace la {
namespace tcn {

using namespace la::tcf;

constexpr int D = 64, M = 64, NE = M + 16, W = D * M + D;
constexpr int NT = 256;  // two warpgroups; two CTAs share an SM
constexpr uint32_t S_ATOM = D * 128;  // 64 state rows x 128 bytes

constexpr uint32_t ID_S = idesc_bf16(128, NE, true, true);   // kf^T [V | 1]
constexpr uint32_t ID_O = idesc_bf16(128, NE, false, true);  // qf [S | Z]

// state kernel shared memory: K tile (fp32, then hi | lo bf16), V tile (fp32,
// then hi | lo bf16) followed by a ones atom and a zeros atom, so that
// [V_hi | 1] and [V_lo | 0] are operands with a 32 KB atom stride.
struct LayA {
    static constexpr uint32_t K = 0, V = 2 * kAtom, ONES = 4 * kAtom, ZEROS = 5 * kAtom;
    static constexpr uint32_t BARS = 6 * kAtom;
    static constexpr uint32_t BYTES = BARS + 64;
    static constexpr uint32_t T_COLS = 128;
};

// read-out kernel shared memory: Q tile (fp32, then hi | lo bf16), state tiles
// [S_hi | Z_hi] and [S_lo | Z_lo] (MN-major, 64 rows, 8 KB atoms) and the fp32
// output staging tile.
struct LayB {
    static constexpr uint32_t Q = 0, S = 2 * kAtom, OUT = 4 * kAtom;
    static constexpr uint32_t BARS = 6 * kAtom;
    static constexpr uint32_t BYTES = BARS + 64;
    static constexpr uint32_t T_COLS = 128;
};

struct NcParams {
    int N, spans, span_len;   // state-kernel spans (the partials' layout)
    int out_spans, out_len;   // read-out spans
    float* part;              // [BH][spans][W]
    unsigned* status;
};

// Byte offset of fp32 element (r, c), c < 64, in a tile of two 32-column atoms.
__device__ __forceinline__ uint32_t f32_off(int r, int c) {
    return (c >> 5) * kAtom + r * 128 + ((((c & 31) >> 2) ^ (r & 7)) << 4) + (c & 3) * 4;
}

__device__ __forceinline__ void split_bf16(float x, float& hi, float& lo) {
    const __nv_bfloat16 h = __float2bfloat16_rn(x);
    hi = __bfloat162float(h);
    lo = x - hi;
}

// In place: the fp32 [128 x 64] tile at `buf` becomes bf16 hi (buf) and lo
// (buf + 16 KB), each one K-major 128-row atom; phi is applied first when PHI,
// and rows >= valid become 0 when ZERO_TAIL.  Each thread reads its
// (row, 8-column) groups before any thread writes.
template <bool PHI, bool ZERO_TAIL>
__device__ __forceinline__ void split_tile(uint8_t* buf, int valid) {
    constexpr int IT = 1024 / NT;  // (row, 8-column) groups per thread
    float x[IT][8];
#pragma unroll
    for (int it = 0; it < IT; ++it) {
        const int item = threadIdx.x + NT * it;
        const int r = item >> 3, j = item & 7;
        const uint4 a = *reinterpret_cast<const uint4*>(buf + f32_off(r, 8 * j));
        const uint4 b = *reinterpret_cast<const uint4*>(buf + f32_off(r, 8 * j + 4));
        x[it][0] = __uint_as_float(a.x);
        x[it][1] = __uint_as_float(a.y);
        x[it][2] = __uint_as_float(a.z);
        x[it][3] = __uint_as_float(a.w);
        x[it][4] = __uint_as_float(b.x);
        x[it][5] = __uint_as_float(b.y);
        x[it][6] = __uint_as_float(b.z);
        x[it][7] = __uint_as_float(b.w);
    }
    __syncthreads();
#pragma unroll
    for (int it = 0; it < IT; ++it) {
        const int item = threadIdx.x + NT * it;
        const int r = item >> 3, j = item & 7;
        uint32_t h[4], l[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            float v0 = x[it][2 * u], v1 = x[it][2 * u + 1];
            if (PHI) {
                v0 = phi_fast(v0);
                v1 = phi_fast(v1);
            }
            if (ZERO_TAIL && r >= valid) v0 = v1 = 0.f;
            float h0, l0, h1, l1;
            split_bf16(v0, h0, l0);
            split_bf16(v1, h1, l1);
            h[u] = pack_bf16(h0, h1);
            l[u] = pack_bf16(l0, l1);
        }
        *reinterpret_cast<uint4*>(buf + swz(r, j)) = make_uint4(h[0], h[1], h[2], h[3]);
        *reinterpret_cast<uint4*>(buf + kAtom + swz(r, j)) = make_uint4(l[0], l[1], l[2], l[3]);
    }
}

__device__ __forceinline__ void sync_tc() {
    fence_proxy_async();
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
}

// ------------------------------------------------------------ state kernel

__global__ void __launch_bounds__(NT, 2)
nc_state_tc_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                   const NcParams p) {
    using Lay = LayA;
    extern __shared__ __align__(1024) uint8_t sm[];
    const int t = threadIdx.x, warp = t >> 5;
    if (smem_u32(sm) & 1023u) {
        if (t == 0) atomicOr(p.status, kErrAlign);
        return;
    }
    uint64_t* tma_bar = reinterpret_cast<uint64_t*>(sm + Lay::BARS);
    uint64_t* mma_bar = tma_bar + 1;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tma_bar + 2);
    volatile int* sh = reinterpret_cast<volatile int*>(tma_bar + 3);
    if (t == 0) {
        mbar_init(tma_bar, 1);
        mbar_init(mma_bar, 1);
        fence_mbar_init();
        sh[1] = 0;
    }
    if (warp == 0) {
        tmem_alloc(tmem_slot, Lay::T_COLS);
        tmem_relinquish();
    }
    for (int i = t; i < static_cast<int>(kAtom / 16); i += NT) {
        reinterpret_cast<uint4*>(sm + Lay::ONES)[i] =
            make_uint4(0x3F803F80u, 0x3F803F80u, 0x3F803F80u, 0x3F803F80u);
        reinterpret_cast<uint4*>(sm + Lay::ZEROS)[i] = make_uint4(0u, 0u, 0u, 0u);
    }
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tm = *tmem_slot;

    const int unit = blockIdx.x;
    const int bh = unit / p.spans, s = unit - bh * p.spans;
    const int n0 = s * p.span_len, n1 = min(p.N, n0 + p.span_len);
    const int nch = (n1 - n0 + L - 1) / L;
    const int q = warp & 3, g = warp >> 2;  // TMEM lane quarter, warpgroup (column half)
    const uint32_t lane = static_cast<uint32_t>(32 * q) << 16;
    const uint32_t sK = smem_u32(sm + Lay::K), sV = smem_u32(sm + Lay::V);
    uint32_t tma_phase = 0, mma_phase = 0;

    auto fail = [&](unsigned code) {
        atomicOr(p.status, code);
        sh[1] = 1;
    };
    auto wait_bar = [&](uint64_t* bar, uint32_t& phase) {
        if (t == 0 && !mbar_wait(bar, phase, kWaitLimit)) fail(kErrWait);
        __syncthreads();
        phase ^= 1u;
    };
    auto load = [&](int c0) {
        mbar_arrive_expect_tx(tma_bar, 4 * kAtom);
        tma_load_3d(sm + Lay::K, &tmK, tma_bar, 0, c0, bh);
        tma_load_3d(sm + Lay::K + kAtom, &tmK, tma_bar, 32, c0, bh);
        tma_load_3d(sm + Lay::V, &tmV, tma_bar, 0, c0, bh);
        tma_load_3d(sm + Lay::V + kAtom, &tmV, tma_bar, 32, c0, bh);
    };

    if (t == 0) load(n0);
    for (int c = 0; c < nch; ++c) {
        const int c0 = n0 + c * L;
        const int valid = min(L, n1 - c0);
        wait_bar(tma_bar, tma_phase);
        split_tile<true, true>(sm + Lay::K, valid);
        split_tile<false, false>(sm + Lay::V, valid);
        sync_tc();
        if (sh[1]) goto cleanup;
        if (t == 0) {
            // K_hi^T [V_hi | 1] + K_hi^T [V_lo | 0] + K_lo^T [V_hi | 1]; the D = 64
            // rows pad to 128 through the A operand's atom stride (rows never read)
#pragma unroll
            for (int k = 0; k < L / 16; ++k)
                mma_bf16(tm, sdesc(sK + 2048 * k, kAtom, 1024), sdesc(sV + 2048 * k, 2 * kAtom, 1024),
                         ID_S, (c > 0 || k > 0) ? 1u : 0u);
#pragma unroll
            for (int k = 0; k < L / 16; ++k)
                mma_bf16(tm, sdesc(sK + 2048 * k, kAtom, 1024),
                         sdesc(sV + kAtom + 2048 * k, 2 * kAtom, 1024), ID_S, 1u);
#pragma unroll
            for (int k = 0; k < L / 16; ++k)
                mma_bf16(tm, sdesc(sK + kAtom + 2048 * k, kAtom, 1024),
                         sdesc(sV + 2048 * k, 2 * kAtom, 1024), ID_S, 1u);
            mma_commit(mma_bar);
        }
        wait_bar(mma_bar, mma_phase);
        fence_after_sync();
        if (t == 0 && c + 1 < nch) load(c0 + L);
    }
    if (q < D / 32) {  // publish the span's [S | Z]: row d < D, this warpgroup's 32 columns
        float* out = p.part + static_cast<size_t>(unit) * W;
        const int d = 32 * q + (t & 31);
        float v[32];
        tmem_ld32(tm + lane + 32 * g, v);
#pragma unroll
        for (int u = 0; u < 8; ++u)
            reinterpret_cast<float4*>(out + d * M + 32 * g)[u] =
                make_float4(v[4 * u], v[4 * u + 1], v[4 * u + 2], v[4 * u + 3]);
        if (g == 0) {
            float z[16];
            tmem_ld16(tm + lane + M, z);
            out[D * M + d] = z[0];
        }
    }

cleanup:
    fence_before_sync();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tm, Lay::T_COLS);
}

// --------------------------------------------------------- read-out kernel

__global__ void __launch_bounds__(NT, 2)
nc_out_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmO,
                 const NcParams p) {
    using Lay = LayB;
    extern __shared__ __align__(1024) uint8_t sm[];
    const int t = threadIdx.x, warp = t >> 5;
    if (smem_u32(sm) & 1023u) {
        if (t == 0) atomicOr(p.status, kErrAlign);
        return;
    }
    uint64_t* tma_bar = reinterpret_cast<uint64_t*>(sm + Lay::BARS);
    uint64_t* mma_bar = tma_bar + 1;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tma_bar + 2);
    volatile int* sh = reinterpret_cast<volatile int*>(tma_bar + 3);
    if (t == 0) {
        mbar_init(tma_bar, 1);
        mbar_init(mma_bar, 1);
        fence_mbar_init();
        sh[1] = 0;
    }
    if (warp == 0) {
        tmem_alloc(tmem_slot, Lay::T_COLS);
        tmem_relinquish();
    }
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tm = *tmem_slot;

    const int unit = blockIdx.x;
    const int bh = unit / p.out_spans, s = unit - bh * p.out_spans;
    const int n0 = s * p.out_len, n1 = min(p.N, n0 + p.out_len);
    const int nch = (n1 - n0 + L - 1) / L;
    const int q = warp & 3, g = warp >> 2;  // TMEM lane quarter, warpgroup (column half)
    const uint32_t lane = static_cast<uint32_t>(32 * q) << 16;
    const uint32_t sQ = smem_u32(sm + Lay::Q), sS = smem_u32(sm + Lay::S);
    uint32_t tma_phase = 0, mma_phase = 0;

    auto fail = [&](unsigned code) {
        atomicOr(p.status, code);
        sh[1] = 1;
    };
    auto wait_bar = [&](uint64_t* bar, uint32_t& phase) {
        if (t == 0 && !mbar_wait(bar, phase, kWaitLimit)) fail(kErrWait);
        __syncthreads();
        phase ^= 1u;
    };
    auto load = [&](int c0) {
        mbar_arrive_expect_tx(tma_bar, 2 * kAtom);
        tma_load_3d(sm + Lay::Q, &tmQ, tma_bar, 0, c0, bh);
        tma_load_3d(sm + Lay::Q + kAtom, &tmQ, tma_bar, 32, c0, bh);
    };
    if (t == 0) load(n0);

    if (q < D / 32) {  // [S | Z] of the head, split into hi and lo MN-major tiles: row d, this
                       // warpgroup's 32 columns (and Z for the first)
        const int d = 32 * q + (t & 31);
        const float* base = p.part + static_cast<size_t>(bh) * p.spans * W;
        for (int j0 = 32 * g; j0 < 32 * g + 32; j0 += 8) {
            float v[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) v[u] = 0.f;
            for (int sp = 0; sp < p.spans; ++sp) {
                const float4* a = reinterpret_cast<const float4*>(base + static_cast<size_t>(sp) * W +
                                                                  d * M + j0);
                const float4 x0 = __ldcg(a), x1 = __ldcg(a + 1);
                v[0] += x0.x;
                v[1] += x0.y;
                v[2] += x0.z;
                v[3] += x0.w;
                v[4] += x1.x;
                v[5] += x1.y;
                v[6] += x1.z;
                v[7] += x1.w;
            }
            uint32_t h[4], l[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                float h0, l0, h1, l1;
                split_bf16(v[2 * u], h0, l0);
                split_bf16(v[2 * u + 1], h1, l1);
                h[u] = pack_bf16(h0, h1);
                l[u] = pack_bf16(l0, l1);
            }
            *reinterpret_cast<uint4*>(sm + Lay::S + swz(d, j0 >> 3)) = make_uint4(h[0], h[1], h[2], h[3]);
            *reinterpret_cast<uint4*>(sm + Lay::S + 2 * S_ATOM + swz(d, j0 >> 3)) =
                make_uint4(l[0], l[1], l[2], l[3]);
        }
        if (g == 0) {
            float z = 0.f;
            for (int sp = 0; sp < p.spans; ++sp) z += __ldcg(base + static_cast<size_t>(sp) * W + D * M + d);
            float zh, zl;
            split_bf16(z, zh, zl);
            const uint32_t ph = pack_bf16(zh, zh), pl = pack_bf16(zl, zl);
            const uint4 hz = make_uint4(ph, ph, ph, ph), lz = make_uint4(pl, pl, pl, pl);
            *reinterpret_cast<uint4*>(sm + Lay::S + S_ATOM + swz(d, 0)) = hz;
            *reinterpret_cast<uint4*>(sm + Lay::S + S_ATOM + swz(d, 1)) = hz;
            *reinterpret_cast<uint4*>(sm + Lay::S + 3 * S_ATOM + swz(d, 0)) = lz;
            *reinterpret_cast<uint4*>(sm + Lay::S + 3 * S_ATOM + swz(d, 1)) = lz;
        }
    }

    for (int c = 0; c < nch; ++c) {
        const int c0 = n0 + c * L;
        wait_bar(tma_bar, tma_phase);
        split_tile<true, false>(sm + Lay::Q, L);
        if (t == 0) tma_store_wait_read();  // the staging tile is free again
        sync_tc();
        if (sh[1]) goto cleanup;
        if (t == 0) {
            // Q_hi [S_hi | Z_hi] + Q_hi [S_lo | Z_lo] + Q_lo [S_hi | Z_hi]
#pragma unroll
            for (int k = 0; k < D / 16; ++k)
                mma_bf16(tm, sdesc(sQ + 32 * k, 16, 1024), sdesc(sS + 2048 * k, S_ATOM, 1024), ID_O,
                         k > 0 ? 1u : 0u);
#pragma unroll
            for (int k = 0; k < D / 16; ++k)
                mma_bf16(tm, sdesc(sQ + 32 * k, 16, 1024),
                         sdesc(sS + 2 * S_ATOM + 2048 * k, S_ATOM, 1024), ID_O, 1u);
#pragma unroll
            for (int k = 0; k < D / 16; ++k)
                mma_bf16(tm, sdesc(sQ + kAtom + 32 * k, 16, 1024), sdesc(sS + 2048 * k, S_ATOM, 1024),
                         ID_O, 1u);
            mma_commit(mma_bar);
        }
        wait_bar(mma_bar, mma_phase);
        fence_after_sync();
        if (t == 0 && c + 1 < nch) load(c0 + L);  // the Q tile is consumed
        {   // V' = num / den, this warpgroup's 32 columns, fp32 into the swizzled staging tile
            const int i = 32 * q + (t & 31);
            float dz[16];
            tmem_ld16(tm + lane + M, dz);
            const float inv = 1.f / dz[0];
            float v[32];
            tmem_ld32(tm + lane + 32 * g, v);
#pragma unroll
            for (int u = 0; u < 8; ++u)
                *reinterpret_cast<float4*>(sm + Lay::OUT + f32_off(i, 32 * g + 4 * u)) =
                    make_float4(v[4 * u] * inv, v[4 * u + 1] * inv, v[4 * u + 2] * inv,
                                v[4 * u + 3] * inv);
        }
        sync_tc();
        if (t == 0) {
            tma_store_3d(&tmO, sm + Lay::OUT, 0, c0, bh);
            tma_store_3d(&tmO, sm + Lay::OUT + kAtom, 32, c0, bh);
            tma_store_commit();
        }
    }

cleanup:
    if (t == 0) tma_store_wait_all();
    fence_before_sync();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tm, Lay::T_COLS);
}

// Spans for a grid of independent (head, span) units: fewest waves x chunks,
// at most 8 spans per head (every read-out CTA sums all of its head's state
// partials, so their number stays small), fewest spans on ties.
inline int spans_for(int BH, int chunks, int slots) {
    int best = 1;
    long best_cost = -1;
    for (int s = 1; s <= std::min(chunks, 8); ++s) {
        const int per = (chunks + s - 1) / s;
        const int eff = (chunks + per - 1) / per;
        const long waves = (static_cast<long>(BH) * eff + slots - 1) / slots;
        const long cost = waves * per;
        if (best_cost < 0 || cost < best_cost) {
            best_cost = cost;
            best = eff;
        }
    }
    return best;
}

// State-kernel spans of a head and their length in tokens.
inline void nc_spans(int BH, int N, int num_sms, int* spans, int* span_len) {
    const int chunks = (N + L - 1) / L;
    const int s = spans_for(BH, chunks, 2 * num_sms);
    *span_len = ((chunks + s - 1) / s) * L;
    *spans = (N + *span_len - 1) / *span_len;
}

}  // namespace tcn

size_t noncausal_forward_tc_f32_scratch(int BH, int N, int num_sms) {
    int spans = 1, len = 0;
    tcn::nc_spans(BH, N, num_sms, &spans, &len);
    return sizeof(float) * static_cast<size_t>(BH) * spans * tcn::W;
}

cudaError_t noncausal_forward_tc_f32(const LaunchCtx& c, const float* Q, const float* K,
                                     const float* V, float* O, int BH, int N) {
    using namespace tcn;
    auto ka = nc_state_tc_kernel;
    auto kb = nc_out_tc_kernel;
    cudaError_t e;
    if ((e = cudaFuncSetAttribute(ka, cudaFuncAttributeMaxDynamicSharedMemorySize, LayA::BYTES)) ||
        (e = cudaFuncSetAttribute(kb, cudaFuncAttributeMaxDynamicSharedMemorySize, LayB::BYTES)) ||
        (e = cudaFuncSetAttribute(ka, cudaFuncAttributePreferredSharedMemoryCarveout,
                                  cudaSharedmemCarveoutMaxShared)) ||
        (e = cudaFuncSetAttribute(kb, cudaFuncAttributePreferredSharedMemoryCarveout,
                                  cudaSharedmemCarveoutMaxShared)))
        return e;
    NcParams p;
    p.N = N;
    nc_spans(BH, N, c.num_sms, &p.spans, &p.span_len);
    const int chunks = (N + L - 1) / L;
    const int slots = 2 * c.num_sms;  // two CTAs per SM (96 KB, 128 TMEM columns each)
    p.out_spans = spans_for(BH, chunks, slots);
    p.out_len = ((chunks + p.out_spans - 1) / p.out_spans) * L;
    p.out_spans = (N + p.out_len - 1) / p.out_len;
    p.status = c.status_word;
    const size_t part_bytes = noncausal_forward_tc_f32_scratch(BH, N, c.num_sms);
    if ((e = scratch_alloc(c, reinterpret_cast<void**>(&p.part), part_bytes)) != cudaSuccess) return e;
    do {
        CUtensorMap mQ, mK, mV, mO;
        if ((e = make_map_f32(&mQ, Q, BH, N, D)) || (e = make_map_f32(&mK, K, BH, N, D)) ||
            (e = make_map_f32(&mV, V, BH, N, M)) || (e = make_map_f32(&mO, O, BH, N, M)))
            break;
        ka<<<BH * p.spans, NT, LayA::BYTES, c.stream>>>(mK, mV, p);
        kb<<<BH * p.out_spans, NT, LayB::BYTES, c.stream>>>(mQ, mO, p);
        note_launch(2);
        e = cudaGetLastError();
    } while (0);
    scratch_free(c, p.part);
    return e;
}

}  // namespace la
