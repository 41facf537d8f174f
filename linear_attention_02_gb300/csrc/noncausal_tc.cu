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
// the lo parts are about 2^-17 of |a b|), accumulated in fp32 in TMEM.  In the
// read-out and the backward, a Z block appended to S (or a ones block to V)
// carries the normaliser through the same products.
//
//   state kernel   one CTA per (head, span): TMA loads fp32 K, V tiles of 64
//                  tokens into a ring of three slots; phi and the split are
//                  done in place (the fp32 tile becomes its hi and lo bf16
//                  tiles); the MMAs accumulate S for the span and the CUDA
//                  cores sum Z; [S | Z] is published as fp32 partials;
//   read-out kernel one CTA per (head, span): sums the partials of the head,
//                  splits [S | Z] into bf16 hi and lo state tiles, then per
//                  chunk loads fp32 Q, applies phi and the split (into an
//                  operand tile, so that the next chunk's copy lands under
//                  this chunk's products), takes the three products into TMEM
//                  and stores num / den as fp32.
// Each input is read once from HBM and the output written once.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <utility>

#include "la_launch.h"
#include "la_plan.h"
#include "tc_common.cuh"

namespace la {
namespace tcn {

using namespace la::tcf;

constexpr int D = 64, M = 64, NE = M + 16, W = D * M + D;
constexpr int NT = 256;  // two warpgroups; two CTAs share an SM
constexpr uint32_t S_ATOM = D * 128;  // 64 state rows x 128 bytes

constexpr uint32_t ID_S = idesc_bf16(128, NE, true, true);   // MN-major x MN-major, N = M + 16
constexpr uint32_t ID_O = idesc_bf16(128, NE, false, true);  // qf [S | Z]

// state kernel shared memory: a ring of three 64-token stages, each an fp32 K
// tile and an fp32 V tile of two 8 KB atoms (32 columns of 64 rows); after the
// split in place each tile is its hi atom followed by its lo atom.
constexpr int LS = 64;                  // tokens per state-kernel stage
constexpr int NSTG = 3;                 // stages in the ring
constexpr uint32_t kAtomS = LS * 128;   // one 64-row atom column
constexpr uint32_t ID_SV = idesc_bf16(128, M, true, true);  // kf^T V, MN-major x MN-major
struct LayA {
    static constexpr uint32_t STAGE = 4 * kAtomS;  // K then V
    static constexpr uint32_t V = 2 * kAtomS;      // V within a stage
    static constexpr uint32_t BARS = NSTG * STAGE;  // copy, split and product barriers, TMEM slot, flags
    static constexpr uint32_t BYTES = BARS + 128;
    static constexpr uint32_t T_COLS = 64;
};
constexpr int NTS = NT + 32;  // state kernel: eight split warps and one issuing warp
static_assert(LayA::BYTES <= 113 * 1024, "two CTAs per SM");

// read-out kernel shared memory: the fp32 Q tile (the copy's landing place),
// the operand tile (Q's hi | lo bf16 atoms, then the fp32 output staging), and
// the state tiles [S_hi | Z_hi] and [S_lo | Z_lo] (MN-major, 64 rows, 8 KB
// atoms).  The split reads Q into registers and writes the operand tile, so
// the next chunk's copy can land while this chunk is multiplied and stored.
struct LayB {
    static constexpr uint32_t Q = 0, S = 2 * kAtom, OP = 4 * kAtom;
    static constexpr uint32_t BARS = 6 * kAtom;
    static constexpr uint32_t BYTES = BARS + 64;
    static constexpr uint32_t T_COLS = 128;
};

// Programmatic dependent launch.  launch_dependents: this CTA lets the next
// kernel in the stream (launched with programmatic stream serialization) start
// its CTAs; dependency_wait: blocks until the preceding kernel in the stream
// has completed and its memory is visible (a no-op when this kernel was not
// launched that way).
__device__ __forceinline__ void pdl_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_dependency_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

struct NcParams {
    int N, spans, span_len;   // state-kernel spans (the partials' layout)
    int out_spans, out_len;   // read-out spans
    float* part;              // [BH][spans][W]
    unsigned* status;
};

// Byte offset of fp32 element (r, c), c < 64, in a tile of two 32-column atoms
// of `atom` bytes each.
__device__ __forceinline__ uint32_t f32_off(int r, int c, uint32_t atom = kAtom) {
    return (c >> 5) * atom + r * 128 + ((((c & 31) >> 2) ^ (r & 7)) << 4) + (c & 3) * 4;
}

// Two values at once: hi = their bf16 pair (one rounding convert), lo = the bf16 pair of
// x - hi (hi unpacked by shift and mask); the same bits as split_bf16 on each.
__device__ __forceinline__ void split_pair(float x0, float x1, uint32_t& hi, uint32_t& lo) {
    hi = pack_bf16(x0, x1);
    lo = pack_bf16(x0 - __uint_as_float(hi << 16), x1 - __uint_as_float(hi & 0xFFFF0000u));
}

__device__ __forceinline__ void split_bf16(float x, float& hi, float& lo) {
    const __nv_bfloat16 h = __float2bfloat16_rn(x);
    hi = __bfloat162float(h);
    lo = x - hi;
}

// In place: the fp32 [128 x 64] tile at `buf` becomes bf16 hi (buf) and lo
// (buf + 16 KB), each one K-major 128-row atom; phi is applied first when PHI,
// and rows >= valid become 0 when ZERO_TAIL.  Thread t takes the 8-column
// group t % 8 of rows t / 8 + (NTH / 8) i, so the eight threads of a row are
// one warp and the hi and lo words written over a row's fp32 values are that
// row's: the warp reads all of its rows before it writes, with no block-wide
// barrier.
template <bool PHI, bool ZERO_TAIL, int NTH = NT>
__device__ __forceinline__ void split_tile(uint8_t* buf, int valid) {
    constexpr int IT = 1024 / NTH;  // (row, 8-column) groups per thread
    float x[IT][8];
#pragma unroll
    for (int it = 0; it < IT; ++it) {
        const int item = threadIdx.x + NTH * it;
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
    __syncwarp();  // a row's reads and writes are all this warp's
#pragma unroll
    for (int it = 0; it < IT; ++it) {
        const int item = threadIdx.x + NTH * it;
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
            split_pair(v0, v1, h[u], l[u]);
        }
        *reinterpret_cast<uint4*>(buf + swz(r, j)) = make_uint4(h[0], h[1], h[2], h[3]);
        *reinterpret_cast<uint4*>(buf + kAtom + swz(r, j)) = make_uint4(l[0], l[1], l[2], l[3]);
    }
}

// split_tile on one 64-row stage, by the NT threads 0 .. NT - 1: the fp32
// [64 x 64] tile at `buf` becomes bf16 hi (buf) and lo (buf + 8 KB), phi applied
// first when PHI.  Thread t takes the 8-column group t % 8 of rows t / 8 and
// t / 8 + NT / 8, so the eight threads of a row are one warp, and the hi and lo
// words written over a row's fp32 values are that row's: no thread outside
// the warp reads them, and the warp needs no block-wide barrier.  With ZSUM, rows >=
// valid become 0 and each thread adds its values to z: the same 8 columns,
// 8 (t % 8) on, in every row it takes.
template <bool PHI, bool ZSUM>
__device__ __forceinline__ void split_stage(uint8_t* buf, int valid, float (&z)[8]) {
    constexpr int IT = LS * 8 / NT;  // rows per thread
    const int j = threadIdx.x & 7;
    float x[IT][8];
#pragma unroll
    for (int it = 0; it < IT; ++it) {
        const int r = (threadIdx.x >> 3) + (NT / 8) * it;
        const uint4 a = *reinterpret_cast<const uint4*>(buf + f32_off(r, 8 * j, kAtomS));
        const uint4 b = *reinterpret_cast<const uint4*>(buf + f32_off(r, 8 * j + 4, kAtomS));
        x[it][0] = __uint_as_float(a.x);
        x[it][1] = __uint_as_float(a.y);
        x[it][2] = __uint_as_float(a.z);
        x[it][3] = __uint_as_float(a.w);
        x[it][4] = __uint_as_float(b.x);
        x[it][5] = __uint_as_float(b.y);
        x[it][6] = __uint_as_float(b.z);
        x[it][7] = __uint_as_float(b.w);
    }
    __syncwarp();  // a row's reads and writes are all this warp's
#pragma unroll
    for (int it = 0; it < IT; ++it) {
        const int r = (threadIdx.x >> 3) + (NT / 8) * it;
        uint32_t h[4], l[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            float v0 = x[it][2 * u], v1 = x[it][2 * u + 1];
            if (PHI) {
                v0 = phi_fast(v0);
                v1 = phi_fast(v1);
            }
            if (ZSUM) {
                v0 = r < valid ? v0 : 0.f;
                v1 = r < valid ? v1 : 0.f;
                z[2 * u] += v0;
                z[2 * u + 1] += v1;
            }
            split_pair(v0, v1, h[u], l[u]);
        }
        *reinterpret_cast<uint4*>(buf + swz(r, j)) = make_uint4(h[0], h[1], h[2], h[3]);
        *reinterpret_cast<uint4*>(buf + kAtomS + swz(r, j)) = make_uint4(l[0], l[1], l[2], l[3]);
    }
}

__device__ __forceinline__ void sync_tc() {
    fence_proxy_async();
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
}

// ------------------------------------------------------------ state kernel
//
// The span's 64-token stages go through a ring of three slots.  Eight warps
// split each stage in place (phi(K) and K, V into hi and lo), each on its own
// rows with no block-wide barrier, and hand it over through the slot's split
// barrier (one arrival per thread); a ninth warp issues the copies and the
// products (S = kf^T V as hi hi + hi lo + lo hi, N = 64) and refills a slot
// with the stage three ahead as soon as the products that read it are done,
// so the split warps wait neither for copies in steady state nor for the
// products.  Z is the sum of the phi(K) rows, added up in fp32 on the CUDA
// cores during the split.

__global__ void __launch_bounds__(NTS, 2)
nc_state_tc_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                   const NcParams p) {
    using Lay = LayA;
    extern __shared__ __align__(1024) uint8_t sm[];
    const int t = threadIdx.x, warp = t >> 5;
    if (smem_u32(sm) & 1023u) {
        if (t == 0) atomicOr(p.status, kErrAlign);
        return;
    }
    uint64_t* full = reinterpret_cast<uint64_t*>(sm + Lay::BARS);  // [NSTG] copy landed
    uint64_t* done = full + NSTG;                                   // [NSTG] split written
    uint64_t* mmab = full + 2 * NSTG;                               // [NSTG] products done
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(full + 3 * NSTG);
    volatile int* sh = reinterpret_cast<volatile int*>(full + 3 * NSTG + 1);
    if (t == 0) {
        for (int b = 0; b < NSTG; ++b) {
            mbar_init(full + b, 1);
            mbar_init(done + b, NT);
            mbar_init(mmab + b, 1);
        }
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
    pdl_launch_dependents();  // the read-out's CTAs may take free slots and start their copies

    const int unit = blockIdx.x;
    const int bh = unit / p.spans, s = unit - bh * p.spans;
    const int n0 = s * p.span_len, n1 = min(p.N, n0 + p.span_len);
    const int nst = max(0, (n1 - n0 + LS - 1) / LS);
    const int q = warp & 3, g = (warp >> 2) & 1;  // TMEM lane quarter, column half (split warps)
    const uint32_t lane = static_cast<uint32_t>(32 * q) << 16;
    float z[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) z[u] = 0.f;

    auto fail = [&](unsigned code) {
        atomicOr(p.status, code);
        sh[1] = 1;
    };

    if (warp == NT / 32) {
        if (t == NT) {  // the issuing thread; a slot's barriers see stage st with parity (st / NSTG) & 1
            int loaded = 0, issued = 0;
            auto load = [&](int st) {
                uint8_t* buf = sm + (st % NSTG) * Lay::STAGE;
                uint64_t* bar = full + st % NSTG;
                const int y = n0 + st * LS;
                mbar_arrive_expect_tx(bar, Lay::STAGE);
                tma_load_3d(buf, &tmK, bar, 0, y, bh);
                tma_load_3d(buf + kAtomS, &tmK, bar, 32, y, bh);
                tma_load_3d(buf + Lay::V, &tmV, bar, 0, y, bh);
                tma_load_3d(buf + Lay::V + kAtomS, &tmV, bar, 32, y, bh);
                ++loaded;
            };
            for (int st = 0; st < min(NSTG, nst); ++st) load(st);
            for (int c = 0; c < nst; ++c) {
                const int w = mbar_wait_or(done + c % NSTG, (c / NSTG) & 1u, kWaitLimit, sh + 1);
                if (w) {
                    if (w == 2) fail(kErrWait);
                    break;
                }
                fence_after_sync();
                // K_hi^T V_hi + K_hi^T V_lo + K_lo^T V_hi; the D = 64 rows of kf^T pad to the
                // MMA's 128 through the A operand's atom stride (accumulator lanes never read)
                const uint32_t sK = smem_u32(sm + (c % NSTG) * Lay::STAGE), sV = sK + Lay::V;
#pragma unroll
                for (int k = 0; k < LS / 16; ++k)
                    mma_bf16(tm, sdesc(sK + 2048 * k, kAtomS, 1024), sdesc(sV + 2048 * k, kAtomS, 1024),
                             ID_SV, (c > 0 || k > 0) ? 1u : 0u);
#pragma unroll
                for (int k = 0; k < LS / 16; ++k)
                    mma_bf16(tm, sdesc(sK + 2048 * k, kAtomS, 1024),
                             sdesc(sV + kAtomS + 2048 * k, kAtomS, 1024), ID_SV, 1u);
#pragma unroll
                for (int k = 0; k < LS / 16; ++k)
                    mma_bf16(tm, sdesc(sK + kAtomS + 2048 * k, kAtomS, 1024),
                             sdesc(sV + 2048 * k, kAtomS, 1024), ID_SV, 1u);
                mma_commit(mmab + c % NSTG);
                ++issued;
                if (c >= 1 && c - 1 + NSTG < nst) {  // stage c - 1's slot, once its products are done
                    const int pv = c - 1;
                    if (!mbar_wait(mmab + pv % NSTG, (pv / NSTG) & 1u, kWaitLimit)) {
                        fail(kErrWait);
                        break;
                    }
                    load(pv + NSTG);
                }
            }
            // the last commit covers every product before it; then every copy still in flight
            // (only the last one into each slot can be: the earlier ones were split)
            if (issued > 0 &&
                !mbar_wait(mmab + (issued - 1) % NSTG, ((issued - 1) / NSTG) & 1u, kWaitLimit))
                fail(kErrWait);
            for (int st = max(0, loaded - NSTG); st < loaded; ++st)
                mbar_wait(full + st % NSTG, (st / NSTG) & 1u, kWaitLimit);
        }
        __syncwarp();
    } else {
        for (int c = 0; c < nst; ++c) {  // every split thread waits for the copy itself
            uint8_t* buf = sm + (c % NSTG) * Lay::STAGE;
            const int w = mbar_wait_or(full + c % NSTG, (c / NSTG) & 1u, kWaitLimit, sh + 1);
            if (w) {
                if (w == 2) fail(kErrWait);
                break;
            }
            const int valid = min(LS, n1 - (n0 + c * LS));
            split_stage<true, true>(buf, valid, z);
            split_stage<false, false>(buf + Lay::V, valid, z);
            fence_proxy_async();
            mbar_arrive(done + c % NSTG);
        }
        // Z: the threads of an 8-column group are the lanes l, l ^ 8, l ^ 16, l ^ 24 of every warp
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            z[u] += __shfl_xor_sync(0xffffffffu, z[u], 8);
            z[u] += __shfl_xor_sync(0xffffffffu, z[u], 16);
        }
    }
    __syncthreads();  // every product is done (or the CTA gives up): slot 0 takes the warps' Z sums
    if (sh[1]) goto cleanup;
    fence_after_sync();
    {
        float* zw = reinterpret_cast<float*>(sm);  // [NT / 32][D]
        if (warp < NT / 32 && (t & 31) < 8) {
#pragma unroll
            for (int u = 0; u < 8; ++u) zw[warp * D + 8 * (t & 31) + u] = z[u];
        }
        __syncthreads();
        float* out = p.part + static_cast<size_t>(unit) * W;
        if (warp < NT / 32 && q < D / 32) {  // publish the span's S: row d < D, 32 columns
            const int d = 32 * q + (t & 31);
            float v[32];
            tmem_ld32(tm + lane + 32 * g, v);
            if (nst == 0)
#pragma unroll
                for (int u = 0; u < 32; ++u) v[u] = 0.f;
#pragma unroll
            for (int u = 0; u < 8; ++u)
                reinterpret_cast<float4*>(out + d * M + 32 * g)[u] =
                    make_float4(v[4 * u], v[4 * u + 1], v[4 * u + 2], v[4 * u + 3]);
        }
        if (t < D) {
            float zz = 0.f;
#pragma unroll
            for (int w = 0; w < NT / 32; ++w) zz += zw[w * D + t];
            out[D * M + t] = zz;
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
    const uint32_t sQ = smem_u32(sm + Lay::OP), sS = smem_u32(sm + Lay::S);  // sQ: the operand tile
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
    bool in_flight = false;  // thread 0: a Q copy not yet waited for, and its phase
    uint32_t ld_phase = 0;
    auto load = [&](int c0) {
        mbar_arrive_expect_tx(tma_bar, 2 * kAtom);
        tma_load_3d(sm + Lay::Q, &tmQ, tma_bar, 0, c0, bh);
        tma_load_3d(sm + Lay::Q + kAtom, &tmQ, tma_bar, 32, c0, bh);
        in_flight = true;
        ld_phase = tma_phase;
    };
    if (t == 0) load(n0);
    pdl_dependency_wait();  // the state kernel's partials are complete (Q does not depend on it)

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
            for (int u = 0; u < 4; ++u) split_pair(v[2 * u], v[2 * u + 1], h[u], l[u]);
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
        if (sh[1]) goto cleanup;
        if (t == 0) in_flight = false;
        {   // phi(Q) split into the operand tile: this thread's (row, 8-column) groups into
            // registers, the Q tile handed back to the next copy, then the hi | lo words
            constexpr int IT = 1024 / NT;
            float x[IT][8];
#pragma unroll
            for (int it = 0; it < IT; ++it) {
                const int r = (t >> 3) + (NT / 8) * it, j = t & 7;
                const uint4 a = *reinterpret_cast<const uint4*>(sm + Lay::Q + f32_off(r, 8 * j));
                const uint4 b = *reinterpret_cast<const uint4*>(sm + Lay::Q + f32_off(r, 8 * j + 4));
                x[it][0] = __uint_as_float(a.x);
                x[it][1] = __uint_as_float(a.y);
                x[it][2] = __uint_as_float(a.z);
                x[it][3] = __uint_as_float(a.w);
                x[it][4] = __uint_as_float(b.x);
                x[it][5] = __uint_as_float(b.y);
                x[it][6] = __uint_as_float(b.z);
                x[it][7] = __uint_as_float(b.w);
            }
            if (t == 0) tma_store_wait_read();  // the last chunk's output has left the operand tile
            __syncthreads();                    // every Q read is done
            if (t == 0 && c + 1 < nch) load(c0 + L);
#pragma unroll
            for (int it = 0; it < IT; ++it) {
                const int r = (t >> 3) + (NT / 8) * it, j = t & 7;
                uint32_t hh[4], ll[4];
#pragma unroll
                for (int u = 0; u < 4; ++u)
                    split_pair(phi_fast(x[it][2 * u]), phi_fast(x[it][2 * u + 1]), hh[u], ll[u]);
                *reinterpret_cast<uint4*>(sm + Lay::OP + swz(r, j)) = make_uint4(hh[0], hh[1], hh[2], hh[3]);
                *reinterpret_cast<uint4*>(sm + Lay::OP + kAtom + swz(r, j)) =
                    make_uint4(ll[0], ll[1], ll[2], ll[3]);
            }
        }
        sync_tc();
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
        if (sh[1]) goto cleanup;
        {   // V' = num / den, this warpgroup's 32 columns, fp32 over the consumed operand tile
            const int i = 32 * q + (t & 31);
            float dz[16];
            tmem_ld16(tm + lane + M, dz);
            const float inv = 1.f / dz[0];
            float v[32];
            tmem_ld32(tm + lane + 32 * g, v);
#pragma unroll
            for (int u = 0; u < 8; ++u)
                *reinterpret_cast<float4*>(sm + Lay::OP + f32_off(i, 32 * g + 4 * u)) =
                    make_float4(v[4 * u] * inv, v[4 * u + 1] * inv, v[4 * u + 2] * inv,
                                v[4 * u + 3] * inv);
        }
        sync_tc();
        if (t == 0) {
            tma_store_3d(&tmO, sm + Lay::OP, 0, c0, bh);
            tma_store_3d(&tmO, sm + Lay::OP + kAtom, 32, c0, bh);
            tma_store_commit();
        }
    }

cleanup:
    if (t == 0) {  // a copy still in flight after an early exit lands before the CTA leaves
        if (in_flight) mbar_wait(tma_bar, ld_phase, kWaitLimit);
        tma_store_wait_all();
    }
    fence_before_sync();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tm, Lay::T_COLS);
}

// ---------------------------------------------------------------- backward
//
// Gradient of the non-causal form for fp32 storage at D = M = 64 ("Transformers
// are RNNs" section 二, eq. linear; the gradients of section 三（一）4 with the
// prefix and suffix sums over all tokens; the denominator by the quotient rule):
//   gn_i = G_i / den_i,  gd_i = -(G_i . O_i) / den_i,  g = [gn | gd 0 .. 0]
//   dqf = g [S | Z]^T                 (query side, with S, Z from the state kernel)
//   [R | r] = sum_i qf_i^T g_i        (query side, per-span partials)
//   dkf = [V | 1] [R | r]^T,  dV = kf R   (key side)
// on the same split-bf16 products as the forward (hi hi + hi lo + lo hi).

constexpr uint32_t ID_DQ = idesc_bf16(128, D, false, false);  // g [S | Z]^T, K-major x K-major
constexpr uint32_t ID_DV = idesc_bf16(128, M, false, true);   // kf R, K-major x MN-major

// K-major descriptor for K step k of a tile whose 64-column atoms are `atom` bytes apart.
__device__ __forceinline__ uint64_t kdesc(uint32_t base, int k, uint32_t atom) {
    return sdesc(base + (k >> 2) * atom + 32 * (k & 3), 16, 1024);
}
// MN-major descriptor for K step k (16 rows) of a tile whose atoms are `lbo` bytes apart.
__device__ __forceinline__ uint64_t mdesc(uint32_t base, int k, uint32_t lbo) {
    return sdesc(base + 2048 * k, lbo, 1024);
}

// query-side kernel shared memory: Q (fp32, then phi(Q) hi | lo), G (fp32, then gn
// hi | lo), O (fp32 when given, then the gd atoms hi | lo), the state tiles
// [S_hi | Z_hi | S_lo | Z_lo] and the fp32 dQ staging tile; the gn and gd atoms
// are 2 kAtom apart, the column stride of the 80-wide g operand.
// Query side: Q (fp32, then phi(Q) hi | lo, then the fp32 dQ staging tile), G (fp32,
// then gn hi | lo), one EXT atom holding gd's hi term in 16-byte chunks 0-1 and its lo
// term in 2-3 (the second N / K atom of [gn | gd] for either term, through the
// descriptors' strides), and [S | Z] hi | lo.  112 KB: two CTAs of one warpgroup share an
// SM.  O, when given, is read by each row's thread from global memory (it only enters gd).
struct LayQ {
    static constexpr uint32_t Q = 0, G = 2 * kAtom, EXT = 4 * kAtom, S = 5 * kAtom;
    static constexpr uint32_t OUT = Q;
    static constexpr uint32_t GSTEP = EXT - G;               // gn hi -> gd hi
    static constexpr uint32_t GSTEP_LO = EXT + 32 - (G + kAtom);  // gn lo -> gd lo
    static constexpr uint32_t BARS = 7 * kAtom;
    static constexpr uint32_t BYTES = BARS + 64;
    static constexpr uint32_t T_O = 0, T_DQ = 80, T_R = 144, T_COLS = 256;
};
constexpr int NTQ = 128;  // query-side threads: one per tile row
static_assert(2 * (LayQ::BYTES + 1024) <= 233472u, "two query-side CTAs per SM");
// key-side kernel shared memory: K (fp32, then phi(K) hi | lo), V (fp32, then
// hi | lo), the ones atom (2 kAtom after V_hi: the column stride of [V_hi | 1]),
// the tiles [R_hi | r_hi | R_lo | r_lo] and the fp32 dK and dV staging tiles.
// Key side: the fp32 dK, dV rows are staged over the K, V tiles they come from, once
// the products have read them, so that a CTA takes 112 KB and two CTAs of two
// warpgroups share an SM (the key side's chunks are independent of each other).
struct LayK {
    static constexpr uint32_t K = 0, V = 2 * kAtom, ONES = 4 * kAtom, R = 5 * kAtom;
    static constexpr uint32_t DK = K, DV = V;
    static constexpr uint32_t BARS = 7 * kAtom;
    static constexpr uint32_t BYTES = BARS + 64;
    static constexpr uint32_t T_DK = 0, T_DV = 64, T_COLS = 128;
};
constexpr int NTK = 256;  // key-side threads: two per tile row (one per 32-column half)
static_assert(2 * (LayK::BYTES + 1024) <= 233472u, "two key-side CTAs per SM");
static_assert(LayQ::BYTES <= 227 * 1024 && LayK::BYTES <= 227 * 1024, "shared memory");

struct NcbParams {
    const float* O;       // the forward's output [BH][N][M] (query side, when given)
    int N;
    int s_spans;          // state partials per head (the state kernel's spans)
    int q_spans, q_len;   // query-side spans (the (R | r) partials' layout)
    int k_spans, k_len;   // key-side spans
    const float* spart;   // [BH][s_spans][W]
    float* rpart;         // [BH][q_spans][W]
    unsigned* status;
};

// Sum of the partials sp < n of row d (this warpgroup's 32 columns into v[], the
// extension word returned), read from [.. ][n][W] at `base`.
__device__ __forceinline__ float sum_partials(const float* base, int n, int d, int g, float (&v)[32]) {
#pragma unroll
    for (int u = 0; u < 32; ++u) v[u] = 0.f;
    float z = 0.f;
    for (int sp = 0; sp < n; ++sp) {
        const float4* a = reinterpret_cast<const float4*>(base + static_cast<size_t>(sp) * W + d * M + 32 * g);
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const float4 x = __ldcg(a + u);
            v[4 * u] += x.x;
            v[4 * u + 1] += x.y;
            v[4 * u + 2] += x.z;
            v[4 * u + 3] += x.w;
        }
        z += __ldcg(base + static_cast<size_t>(sp) * W + D * M + d);
    }
    return z;
}

// Row d, columns 32 g .. 32 g + 31 of a state as bf16 hi (at `hi`) and lo (at
// `lo`) swizzled 64-row atoms.
__device__ __forceinline__ void put_state_row(uint8_t* hi, uint8_t* lo, int d, int g, const float (&v)[32]) {
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        uint32_t h[4], l[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) split_pair(v[8 * c + 2 * u], v[8 * c + 2 * u + 1], h[u], l[u]);
        *reinterpret_cast<uint4*>(hi + swz(d, 4 * g + c)) = make_uint4(h[0], h[1], h[2], h[3]);
        *reinterpret_cast<uint4*>(lo + swz(d, 4 * g + c)) = make_uint4(l[0], l[1], l[2], l[3]);
    }
}

// An extension row: x in column 0, zeros in columns 1 .. 15 (hi and lo atoms).
__device__ __forceinline__ void put_ext_row(uint8_t* hi, uint8_t* lo, int r, float x) {
    float h, l;
    split_bf16(x, h, l);
    *reinterpret_cast<uint4*>(hi + swz(r, 0)) = make_uint4(pack_bf16(h, 0.f), 0u, 0u, 0u);
    *reinterpret_cast<uint4*>(hi + swz(r, 1)) = make_uint4(0u, 0u, 0u, 0u);
    *reinterpret_cast<uint4*>(lo + swz(r, 0)) = make_uint4(pack_bf16(l, 0.f), 0u, 0u, 0u);
    *reinterpret_cast<uint4*>(lo + swz(r, 1)) = make_uint4(0u, 0u, 0u, 0u);
}

// phi'(x) = min(phi(x), 1) for 32 columns of row r of a split phi tile (hi at
// `hi`, lo one atom after): phi = hi + lo.
__device__ __forceinline__ void dphi_row(const uint8_t* hi, int r, int g, float (&f)[32]) {
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        const uint4 a = *reinterpret_cast<const uint4*>(hi + swz(r, 4 * g + c));
        const uint4 b = *reinterpret_cast<const uint4*>(hi + kAtom + swz(r, 4 * g + c));
        const uint32_t wa[4] = {a.x, a.y, a.z, a.w}, wb[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            f[8 * c + 2 * u] = fminf(__uint_as_float(wa[u] << 16) + __uint_as_float(wb[u] << 16), 1.f);
            f[8 * c + 2 * u + 1] =
                fminf(__uint_as_float(wa[u] & 0xFFFF0000u) + __uint_as_float(wb[u] & 0xFFFF0000u), 1.f);
        }
    }
}

template <bool HAS_O>
__global__ void __launch_bounds__(NTQ, 2)
ncb_query_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmG,
                    const __grid_constant__ CUtensorMap tmdQ, const NcbParams p) {
    using Lay = LayQ;
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
    const int bh = unit / p.q_spans, s = unit - bh * p.q_spans;
    const int n0 = s * p.q_len, n1 = min(p.N, n0 + p.q_len);
    const int nch = (n1 - n0 + L - 1) / L;
    const int q = warp;  // TMEM lane quarter; one warpgroup: each thread takes its whole row
    const int row = 32 * q + (t & 31);
    const uint32_t lane = static_cast<uint32_t>(32 * q) << 16;
    const uint32_t sQ = smem_u32(sm + Lay::Q), sG = smem_u32(sm + Lay::G), sS = smem_u32(sm + Lay::S);
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
    auto load = [&](int c0) {  // thread 0 only
        mbar_arrive_expect_tx(tma_bar, 4 * kAtom);
        for (int a = 0; a < 2; ++a) {
            tma_load_3d(sm + Lay::Q + a * kAtom, &tmQ, tma_bar, 32 * a, c0, bh);
            tma_load_3d(sm + Lay::G + a * kAtom, &tmG, tma_bar, 32 * a, c0, bh);
        }
    };
    if (t == 0) load(n0);
    pdl_launch_dependents();  // the key side's CTAs may take free slots and start their copies
    pdl_dependency_wait();    // the state pass's partials are complete (Q, G do not depend on it)

    if (q < D / 32) {  // [S | Z] of the head, split: row d, both 32-column halves
      for (int g = 0; g < 2; ++g) {
        float v[32];
        const float z = sum_partials(p.spart + static_cast<size_t>(bh) * p.s_spans * W, p.s_spans, row, g, v);
        put_state_row(sm + Lay::S, sm + Lay::S + 2 * S_ATOM, row, g, v);
        if (g == 0) {  // Z, sixteen copies (the den column of qf [S | Z] reads the first)
            float zh, zl;
            split_bf16(z, zh, zl);
            const uint32_t ph = pack_bf16(zh, zh), pl = pack_bf16(zl, zl);
            for (int c = 0; c < 2; ++c) {
                *reinterpret_cast<uint4*>(sm + Lay::S + S_ATOM + swz(row, c)) = make_uint4(ph, ph, ph, ph);
                *reinterpret_cast<uint4*>(sm + Lay::S + 3 * S_ATOM + swz(row, c)) = make_uint4(pl, pl, pl, pl);
            }
        }
      }
    }

    for (int c = 0; c < nch; ++c) {
        const int c0 = n0 + c * L;
        const int valid = min(L, n1 - c0);
        wait_bar(tma_bar, tma_phase);
        split_tile<true, false, NTQ>(sm + Lay::Q, L);  // phi(Q) hi | lo (rows past N are 0: phi(0) = 1
                                                       // there, but their g rows are 0)
        sync_tc();
        if (sh[1]) goto cleanup;
        if (t == 0) {  // O_ext = qf [S | Z]
#pragma unroll
            for (int k = 0; k < D / 16; ++k)
                mma_bf16(tm + Lay::T_O, sdesc(sQ + 32 * k, 16, 1024), sdesc(sS + 2048 * k, S_ATOM, 1024), ID_O,
                         k > 0 ? 1u : 0u);
#pragma unroll
            for (int k = 0; k < D / 16; ++k)
                mma_bf16(tm + Lay::T_O, sdesc(sQ + 32 * k, 16, 1024),
                         sdesc(sS + 2 * S_ATOM + 2048 * k, S_ATOM, 1024), ID_O, 1u);
#pragma unroll
            for (int k = 0; k < D / 16; ++k)
                mma_bf16(tm + Lay::T_O, sdesc(sQ + kAtom + 32 * k, 16, 1024), sdesc(sS + 2048 * k, S_ATOM, 1024),
                         ID_O, 1u);
            mma_commit(mma_bar);
        }
        float gv[2][32], go = 0.f;
        if (HAS_O && row < valid) {  // G . O of this row: O from global memory, G from the tile
            const float4* orow = reinterpret_cast<const float4*>(p.O + (static_cast<size_t>(bh) * p.N + c0 + row) * M);
#pragma unroll
            for (int h = 0; h < 2; ++h)
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const float4 a = *reinterpret_cast<const float4*>(sm + Lay::G + f32_off(row, 32 * h + 4 * u));
                    const float4 b = __ldg(orow + 8 * h + u);
                    gv[h][4 * u] = a.x;
                    gv[h][4 * u + 1] = a.y;
                    gv[h][4 * u + 2] = a.z;
                    gv[h][4 * u + 3] = a.w;
                    go = fmaf(a.x, b.x, fmaf(a.y, b.y, fmaf(a.z, b.z, fmaf(a.w, b.w, go))));
                }
        } else {
#pragma unroll
            for (int h = 0; h < 2; ++h)
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const float4 a = *reinterpret_cast<const float4*>(sm + Lay::G + f32_off(row, 32 * h + 4 * u));
                    gv[h][4 * u] = a.x;
                    gv[h][4 * u + 1] = a.y;
                    gv[h][4 * u + 2] = a.z;
                    gv[h][4 * u + 3] = a.w;
                }
        }
        wait_bar(mma_bar, mma_phase);
        fence_after_sync();
        float den;
        {
            float dz[16];
            tmem_ld16(tm + lane + Lay::T_O + M, dz);
            den = dz[0];
        }
        const float inv = row < valid ? 1.f / den : 0.f;
        if (!HAS_O) {  // O = num / den, and G . O
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                float ov[32];
                tmem_ld32(tm + lane + Lay::T_O + 32 * h, ov);
#pragma unroll
                for (int u = 0; u < 32; ++u) go = fmaf(gv[h][u], ov[u] * inv, go);
            }
        }
        const float gd = -go * inv;
        __syncthreads();  // every G row is read: the tile takes g from here on
        {   // gn = G / den, split, into the G tile's atoms; gd's two terms into the EXT atom
#pragma unroll
            for (int h = 0; h < 2; ++h) {
#pragma unroll
                for (int u = 0; u < 32; ++u) gv[h][u] *= inv;
                put_state_row(sm + Lay::G, sm + Lay::G + kAtom, row, h, gv[h]);
            }
            float gh, gl;
            split_bf16(gd, gh, gl);
            *reinterpret_cast<uint4*>(sm + Lay::EXT + swz(row, 0)) = make_uint4(pack_bf16(gh, 0.f), 0u, 0u, 0u);
            *reinterpret_cast<uint4*>(sm + Lay::EXT + swz(row, 1)) = make_uint4(0u, 0u, 0u, 0u);
            *reinterpret_cast<uint4*>(sm + Lay::EXT + swz(row, 2)) = make_uint4(pack_bf16(gl, 0.f), 0u, 0u, 0u);
            *reinterpret_cast<uint4*>(sm + Lay::EXT + swz(row, 3)) = make_uint4(0u, 0u, 0u, 0u);
        }
        sync_tc();
        if (t == 0) {
            const uint32_t sGl = sG + kAtom;
            // dqf = g [S | Z]^T: g_hi [S | Z]_hi + g_hi [S | Z]_lo + g_lo [S | Z]_hi
#pragma unroll
            for (int k = 0; k < NE / 16; ++k)
                mma_bf16(tm + Lay::T_DQ, kdesc(sG, k, Lay::GSTEP), kdesc(sS, k, S_ATOM), ID_DQ, k > 0 ? 1u : 0u);
#pragma unroll
            for (int k = 0; k < NE / 16; ++k)
                mma_bf16(tm + Lay::T_DQ, kdesc(sG, k, Lay::GSTEP), kdesc(sS + 2 * S_ATOM, k, S_ATOM), ID_DQ, 1u);
#pragma unroll
            for (int k = 0; k < NE / 16; ++k)
                mma_bf16(tm + Lay::T_DQ, kdesc(sGl, k, Lay::GSTEP_LO), kdesc(sS, k, S_ATOM), ID_DQ, 1u);
            // [R | r] += qf^T g (the D = 64 rows pad to 128 through the A operand's atom stride)
#pragma unroll
            for (int k = 0; k < L / 16; ++k)
                mma_bf16(tm + Lay::T_R, mdesc(sQ, k, kAtom), mdesc(sG, k, Lay::GSTEP), ID_S,
                         (c > 0 || k > 0) ? 1u : 0u);
#pragma unroll
            for (int k = 0; k < L / 16; ++k)
                mma_bf16(tm + Lay::T_R, mdesc(sQ, k, kAtom), mdesc(sGl, k, Lay::GSTEP_LO), ID_S, 1u);
#pragma unroll
            for (int k = 0; k < L / 16; ++k)
                mma_bf16(tm + Lay::T_R, mdesc(sQ + kAtom, k, kAtom), mdesc(sG, k, Lay::GSTEP), ID_S, 1u);
            mma_commit(mma_bar);
        }
        wait_bar(mma_bar, mma_phase);
        fence_after_sync();
        {   // dQ = dqf * phi'(Q) -> fp32 staging tile over the Q tile: phi'(Q) of the whole row
            // is read before any thread writes over it
            float f[2][32];
#pragma unroll
            for (int h = 0; h < 2; ++h) dphi_row(sm + Lay::Q, row, h, f[h]);
            __syncthreads();
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                float v[32];
                tmem_ld32(tm + lane + Lay::T_DQ + 32 * h, v);
#pragma unroll
                for (int u = 0; u < 8; ++u)
                    *reinterpret_cast<float4*>(sm + Lay::OUT + f32_off(row, 32 * h + 4 * u)) =
                        make_float4(v[4 * u] * f[h][4 * u], v[4 * u + 1] * f[h][4 * u + 1],
                                    v[4 * u + 2] * f[h][4 * u + 2], v[4 * u + 3] * f[h][4 * u + 3]);
            }
        }
        sync_tc();
        if (t == 0) {
            tma_store_3d(&tmdQ, sm + Lay::OUT, 0, c0, bh);
            tma_store_3d(&tmdQ, sm + Lay::OUT + kAtom, 32, c0, bh);
            tma_store_commit();
            if (c + 1 < nch) {  // the staged rows are read out of the Q tile first
                tma_store_wait_read();
                load(c0 + L);
            }
        }
    }
    if (q < D / 32) {  // publish this span's [R | r]
        float* out = p.rpart + (static_cast<size_t>(bh) * p.q_spans + s) * W;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            float v[32];
            tmem_ld32(tm + lane + Lay::T_R + 32 * h, v);
#pragma unroll
            for (int u = 0; u < 8; ++u)
                reinterpret_cast<float4*>(out + row * M + 32 * h)[u] =
                    make_float4(v[4 * u], v[4 * u + 1], v[4 * u + 2], v[4 * u + 3]);
        }
        float z[16];
        tmem_ld16(tm + lane + Lay::T_R + M, z);
        out[D * M + row] = z[0];
    }

cleanup:  // the only early exit follows a copy wait: no copy of this CTA is in flight
    if (t == 0) tma_store_wait_all();
    fence_before_sync();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tm, Lay::T_COLS);
}

__global__ void __launch_bounds__(NTK, 2)
ncb_key_tc_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                  const __grid_constant__ CUtensorMap tmdK, const __grid_constant__ CUtensorMap tmdV,
                  const NcbParams p) {
    using Lay = LayK;
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
    for (int i = t; i < static_cast<int>(kAtom / 16); i += NTK)
        reinterpret_cast<uint4*>(sm + Lay::ONES)[i] =
            make_uint4(0x3F803F80u, 0x3F803F80u, 0x3F803F80u, 0x3F803F80u);
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tm = *tmem_slot;

    const int unit = blockIdx.x;
    const int bh = unit / p.k_spans, s = unit - bh * p.k_spans;
    const int n0 = s * p.k_len, n1 = min(p.N, n0 + p.k_len);
    const int nch = (n1 - n0 + L - 1) / L;
    const int q = warp & 3, g = warp >> 2;  // TMEM lane quarter; the row's 32-column half
    const int row = 32 * q + (t & 31);
    const uint32_t lane = static_cast<uint32_t>(32 * q) << 16;
    const uint32_t sK = smem_u32(sm + Lay::K), sV = smem_u32(sm + Lay::V), sR = smem_u32(sm + Lay::R);
    constexpr uint32_t VSTEP = Lay::ONES - Lay::V;  // [V_hi | 1]: the ones atom 2 kAtom after V_hi
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
    auto load = [&](int c0) {  // thread 0 only
        mbar_arrive_expect_tx(tma_bar, 4 * kAtom);
        for (int a = 0; a < 2; ++a) {
            tma_load_3d(sm + Lay::K + a * kAtom, &tmK, tma_bar, 32 * a, c0, bh);
            tma_load_3d(sm + Lay::V + a * kAtom, &tmV, tma_bar, 32 * a, c0, bh);
        }
    };
    if (t == 0) load(n0);
    pdl_dependency_wait();  // the query side's partials are complete (K, V do not depend on it)

    if (q < D / 32) {  // [R | r] of the head (the query side's partials), split: this half
        float v[32];
        const float r = sum_partials(p.rpart + static_cast<size_t>(bh) * p.q_spans * W, p.q_spans, row, g, v);
        put_state_row(sm + Lay::R, sm + Lay::R + 2 * S_ATOM, row, g, v);
        if (g == 0) put_ext_row(sm + Lay::R + S_ATOM, sm + Lay::R + 3 * S_ATOM, row, r);
    }

    for (int c = 0; c < nch; ++c) {
        const int c0 = n0 + c * L;
        wait_bar(tma_bar, tma_phase);
        split_tile<true, false, NTK>(sm + Lay::K, L);   // phi(K) hi | lo
        split_tile<false, false, NTK>(sm + Lay::V, L);  // V hi | lo
        sync_tc();
        if (sh[1]) goto cleanup;
        if (t == 0) {
            const uint32_t sVl = sV + kAtom, sKl = sK + kAtom, sRl = sR + 2 * S_ATOM;
            // dkf = [V | 1] [R | r]^T: [V_hi | 1][R | r]_hi + [V_hi | 1][R | r]_lo + V_lo R_hi
#pragma unroll
            for (int k = 0; k < NE / 16; ++k)
                mma_bf16(tm + Lay::T_DK, kdesc(sV, k, VSTEP), kdesc(sR, k, S_ATOM), ID_DQ, k > 0 ? 1u : 0u);
#pragma unroll
            for (int k = 0; k < NE / 16; ++k)
                mma_bf16(tm + Lay::T_DK, kdesc(sV, k, VSTEP), kdesc(sRl, k, S_ATOM), ID_DQ, 1u);
#pragma unroll
            for (int k = 0; k < M / 16; ++k)
                mma_bf16(tm + Lay::T_DK, kdesc(sVl, k, VSTEP), kdesc(sR, k, S_ATOM), ID_DQ, 1u);
            // dV = kf R: kf_hi R_hi + kf_hi R_lo + kf_lo R_hi
#pragma unroll
            for (int k = 0; k < D / 16; ++k)
                mma_bf16(tm + Lay::T_DV, kdesc(sK, k, kAtom), mdesc(sR, k, S_ATOM), ID_DV, k > 0 ? 1u : 0u);
#pragma unroll
            for (int k = 0; k < D / 16; ++k)
                mma_bf16(tm + Lay::T_DV, kdesc(sK, k, kAtom), mdesc(sRl, k, S_ATOM), ID_DV, 1u);
#pragma unroll
            for (int k = 0; k < D / 16; ++k)
                mma_bf16(tm + Lay::T_DV, kdesc(sKl, k, kAtom), mdesc(sR, k, S_ATOM), ID_DV, 1u);
            mma_commit(mma_bar);
        }
        wait_bar(mma_bar, mma_phase);
        fence_after_sync();
        {   // dK = dkf * phi'(K), dV -> fp32 staging tiles over the K, V tiles, this thread's
            // half row: phi'(K) is read from the K tile before any thread writes over it
            float f[32], v[32];
            dphi_row(sm + Lay::K, row, g, f);
            __syncthreads();
            tmem_ld32(tm + lane + Lay::T_DK + 32 * g, v);
#pragma unroll
            for (int u = 0; u < 8; ++u)
                *reinterpret_cast<float4*>(sm + Lay::DK + f32_off(row, 32 * g + 4 * u)) =
                    make_float4(v[4 * u] * f[4 * u], v[4 * u + 1] * f[4 * u + 1], v[4 * u + 2] * f[4 * u + 2],
                                v[4 * u + 3] * f[4 * u + 3]);
            tmem_ld32(tm + lane + Lay::T_DV + 32 * g, v);
#pragma unroll
            for (int u = 0; u < 8; ++u)
                *reinterpret_cast<float4*>(sm + Lay::DV + f32_off(row, 32 * g + 4 * u)) =
                    make_float4(v[4 * u], v[4 * u + 1], v[4 * u + 2], v[4 * u + 3]);
        }
        sync_tc();
        if (t == 0) {
            for (int a = 0; a < 2; ++a) {
                tma_store_3d(&tmdK, sm + Lay::DK + a * kAtom, 32 * a, c0, bh);
                tma_store_3d(&tmdV, sm + Lay::DV + a * kAtom, 32 * a, c0, bh);
            }
            tma_store_commit();
            if (c + 1 < nch) {  // the staged rows are read out of the input tiles first
                tma_store_wait_read();
                load(c0 + L);
            }
        }
    }

cleanup:  // the only early exit follows a copy wait: no copy of this CTA is in flight
    if (t == 0) tma_store_wait_all();
    fence_before_sync();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tm, Lay::T_COLS);
}

// Launches `kern` so that it may start while the kernel before it in `stream`
// finishes (programmatic stream serialization); the kernel waits for that
// kernel's results itself (pdl_dependency_wait) and only reads inputs that do
// not depend on it before then.  Its CTAs start only after every CTA of the
// kernel before it has started, so none of them can hold a slot it needs.
template <typename... Params, typename... Args>
cudaError_t launch_dependent(void (*kern)(Params...), int grid, int block, uint32_t smem,
                             cudaStream_t stream, Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(block);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
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

// Spans of the backward's query and key kernels: two CTAs per SM.
inline void ncb_spans(int BH, int N, int num_sms, int* spans, int* span_len) {
    const int chunks = (N + L - 1) / L;
    const int s = spans_for(BH, chunks, 2 * num_sms);
    *span_len = ((chunks + s - 1) / s) * L;
    *spans = (N + *span_len - 1) / *span_len;
}

}  // namespace tcn

size_t noncausal_backward_tc_f32_scratch(int BH, int N, int num_sms) {
    int s_spans = 1, q_spans = 1, len = 0;
    tcn::nc_spans(BH, N, num_sms, &s_spans, &len);
    tcn::ncb_spans(BH, N, num_sms, &q_spans, &len);
    return plan::up256(sizeof(float) * static_cast<size_t>(BH) * s_spans * tcn::W) +
           sizeof(float) * static_cast<size_t>(BH) * q_spans * tcn::W;
}

cudaError_t noncausal_backward_tc_f32(const LaunchCtx& c, const float* Q, const float* K,
                                      const float* V, const float* O, const float* G, float* dQ,
                                      float* dK, float* dV, int BH, int N) {
    using namespace tcn;
    auto ka = nc_state_tc_kernel;
    auto kq = O ? ncb_query_tc_kernel<true> : ncb_query_tc_kernel<false>;
    auto kk = ncb_key_tc_kernel;
    cudaError_t e;
    if ((e = cudaFuncSetAttribute(ka, cudaFuncAttributeMaxDynamicSharedMemorySize, LayA::BYTES)) ||
        (e = cudaFuncSetAttribute(kq, cudaFuncAttributeMaxDynamicSharedMemorySize, LayQ::BYTES)) ||
        (e = cudaFuncSetAttribute(kk, cudaFuncAttributeMaxDynamicSharedMemorySize, LayK::BYTES)))
        return e;
    for (const void* f : {reinterpret_cast<const void*>(ka), reinterpret_cast<const void*>(kq),
                          reinterpret_cast<const void*>(kk)})
        if ((e = cudaFuncSetAttribute(f, cudaFuncAttributePreferredSharedMemoryCarveout,
                                      cudaSharedmemCarveoutMaxShared)))
            return e;
    NcParams sp;  // the state kernel's parameters (the forward's state pass)
    sp.N = N;
    nc_spans(BH, N, c.num_sms, &sp.spans, &sp.span_len);
    sp.out_spans = sp.out_len = 0;
    sp.status = c.status_word;
    NcbParams p;
    p.N = N;
    p.s_spans = sp.spans;
    ncb_spans(BH, N, c.num_sms, &p.q_spans, &p.q_len);
    p.k_spans = p.q_spans;
    p.k_len = p.q_len;
    p.O = O;
    p.status = c.status_word;
    char* ws = nullptr;
    if ((e = scratch_alloc(c, reinterpret_cast<void**>(&ws), noncausal_backward_tc_f32_scratch(BH, N, c.num_sms))))
        return e;
    sp.part = reinterpret_cast<float*>(ws);
    p.spart = sp.part;
    p.rpart = reinterpret_cast<float*>(ws + plan::up256(sizeof(float) * static_cast<size_t>(BH) * sp.spans * W));
    do {
        CUtensorMap mQ, mK, mV, mG, mdQ, mdK, mdV, mKs, mVs;
        if ((e = make_map_f32(&mQ, Q, BH, N, D)) || (e = make_map_f32(&mK, K, BH, N, D)) ||
            (e = make_map_f32(&mV, V, BH, N, M)) || (e = make_map_f32(&mG, G, BH, N, M)) ||
            (e = make_map_f32(&mdQ, dQ, BH, N, D)) || (e = make_map_f32(&mdK, dK, BH, N, D)) ||
            (e = make_map_f32(&mdV, dV, BH, N, M)) || (e = make_map_f32(&mKs, K, BH, N, D, LS)) ||
            (e = make_map_f32(&mVs, V, BH, N, M, LS)))
            break;
        ka<<<BH * sp.spans, NTS, LayA::BYTES, c.stream>>>(mKs, mVs, sp);
        // the query and key sides start under the tail of the kernel before them
        // (programmatic dependent launch) and wait for its partials in-kernel
        if ((e = launch_dependent(kq, BH * p.q_spans, NTQ, LayQ::BYTES, c.stream, mQ, mG, mdQ, p)) ||
            (e = launch_dependent(kk, BH * p.k_spans, NTK, LayK::BYTES, c.stream, mK, mV, mdK, mdV, p)))
            break;
        note_launch(3);
        e = cudaGetLastError();
    } while (0);
    scratch_free(c, ws);
    return e;
}

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
        if ((e = make_map_f32(&mQ, Q, BH, N, D)) || (e = make_map_f32(&mK, K, BH, N, D, LS)) ||
            (e = make_map_f32(&mV, V, BH, N, M, LS)) || (e = make_map_f32(&mO, O, BH, N, M)))
            break;
        ka<<<BH * p.spans, NTS, LayA::BYTES, c.stream>>>(mK, mV, p);
        // the read-out starts under the state kernel's tail (programmatic dependent launch):
        // its prologue and first Q copy overlap, and it waits for the partials in-kernel
        if ((e = launch_dependent(kb, BH * p.out_spans, NT, LayB::BYTES, c.stream, mQ, mO, p))) break;
        note_launch(2);
        e = cudaGetLastError();
    } while (0);
    scratch_free(c, p.part);
    return e;
}

}  // namespace la
