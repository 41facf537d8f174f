// poly_tc.cu -- attention with the degree-2 polynomial similarity (q . k)^2 on
// the 5th-generation tensor core, bf16 storage, D = 32, M = 64.
//
// "【论文解读】Transformers are RNNs" section 二 (3) writes (x^T y)^2 as the
// inner product of the explicit feature maps phi(x) = (x_a x_b)_{a,b}, C = D^2
// features, so that
//     V'_i = phi(Q_i)^T S / phi(Q_i)^T Z,  S = sum_j phi(K_j) V_j^T,  Z = sum_j phi(K_j)
// with the sums over j <= i (causal, section 三) or over all j.  With C = 1024
// both contractions are dense products -- phi(Q) [S | Z] (K = C) and the state
// update phi(K)^T [V | 1] (M = C) -- which is what the tensor core is for.
//
// The fp32 state of one head, C x (M + 16) with the ones block that carries Z,
// needs 640 TMEM columns, more than an SM has, so the C features are cut into
// 8 slices of 128 (slice s: a in [4s, 4s + 4), all b) and a CTA owns two
// slices of one head for the whole sequence (4 CTAs per head).  Per chunk of
// 128 tokens a CTA
//   * builds phi(Q) and phi(K) of a slice from the raw Q, K rows (one thread
//     per token, q_a q_b as exact-product bf16 pairs) into swizzled tiles,
//   * takes O_ext += phi(Q)_s [S_s | Z_s] against the state before the chunk,
//     kept as two bf16 terms (hi = bf16(x), lo = bf16(x - hi)), and
//     S_s += phi(K)_s^T [V | 1] into TMEM, for each of its two slices,
//   * (first slice pair only) adds the intra-chunk terms
//     sum_{j <= i, same chunk} (q_i . k_j)^2 [V_j | 1]: P = Q K^T on the
//     tensor core, squared, masked and packed to bf16 in place in TMEM, and
//     P [V | 1] read from there,
//   * copies the updated state to its two bf16 terms for the next chunk, and
//     adds its partial [numerator | normaliser] rows into an fp32 accumulator
//     in global memory with a TMA bulk reduce-add.
// The features take both signs, so (q . k)^2 can be far smaller than the terms
// it sums; one bf16 rounding of S and Z (independent for the numerator and
// the normaliser) then shows in the quotient (3% on a single token), hence the
// two-term state.  The roundings of phi(Q) and phi(K) are common to the
// numerator and the normaliser and cancel in it.
// Without causality the state is built over all chunks first, then read.  A
// last kernel divides and stores bf16.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "la_launch.h"
#include "la_plan.h"
#include "tc_common.cuh"

namespace la {
namespace tpoly {

using namespace la::tcf;

constexpr int D = 32, M = 64, NE = M + 16;
constexpr int FS = 128;               // features per slice
constexpr int NT = 128;               // one thread per token row / TMEM lane
static_assert(plan::kPolyTcGroups * 2 * FS == D * D, "two slices per CTA cover the D^2 features");

// Shared memory, byte offsets from a 1024-aligned base.  The EXT atom holds,
// per 128-byte row, the hi term of Z of the first slice (16-byte chunks 0-1),
// of the second (2-3), bf16 ones (4-5) and the lo term of the first slice's Z
// (6-7); EXT2 chunks 0-1 the lo term of the second's.  They are the second N
// atoms of [S_s | Z_s] (rows = features) and of [V | 1] (rows = tokens),
// reached through the operand descriptors' leading-byte offsets, so they lie
// after the S tiles and V.  The fp32 partial rows are staged over the phi
// tiles, which are idle from the chunk's last product to the next chunk.
struct Lay {
    static constexpr uint32_t QR = 0;               // raw Q rows [128][32] bf16, 64-byte swizzle
    static constexpr uint32_t KR = QR + 8192;       // raw K rows
    static constexpr uint32_t S0 = KR + 8192;       // hi term of S, first slice [128 features][64]
    static constexpr uint32_t S1 = S0 + kAtom;      // of the second
    static constexpr uint32_t S0L = S1 + kAtom;     // lo terms
    static constexpr uint32_t S1L = S0L + kAtom;
    static constexpr uint32_t V = S1L + kAtom;      // V [128][64], 128-byte swizzle
    static constexpr uint32_t EXT = V + kAtom;
    static constexpr uint32_t EXT2 = EXT + kAtom;
    static constexpr uint32_t FQ = EXT2 + kAtom;    // phi(Q) of a slice: [128 tokens][128 features]
    static constexpr uint32_t FK = FQ + 2 * kAtom;  // phi(K) of a slice
    static constexpr uint32_t QP = FK + 2 * kAtom;  // Q, K rows padded to 64 columns (P = Q K^T)
    static constexpr uint32_t KP = QP + kAtom;
    static constexpr uint32_t STG = FQ;  // fp32 partial rows: three [128][32] boxes, 128-byte swizzle
    static constexpr uint32_t BARS = KP + kAtom;
    static constexpr uint32_t BYTES = BARS + 64;
    // tensor memory: S of the two slices, O_ext, P (packed in place to its first 64 columns)
    static constexpr uint32_t T_S0 = 0, T_S1 = NE, T_O = 2 * NE, T_P = 256, T_COLS = 512;
    static_assert(STG + 3 * kAtom <= QP && BYTES <= 227 * 1024, "shared memory");
    static_assert(T_O + NE <= T_P && T_P + L <= T_COLS, "tensor memory");
};

struct PolyParams {
    int N, BH, CH;         // tokens, heads, chunks per head
    int causal;
    unsigned* status;      // device error word
};

// 16-byte chunk c (0 .. 7) of row `row` of the EXT atom, swizzled.
__device__ __forceinline__ uint32_t ext_off(int row, int c) { return Lay::EXT + swz(row, c); }

// 16-byte chunk c (0 .. 3) of row `row` of a [128][32] bf16 tile with the 64-byte swizzle.
__device__ __forceinline__ uint32_t swz64(int row, int c) { return row * 64 + ((c ^ ((row >> 1) & 3)) << 4); }

// TMA bulk reduce-add of an fp32 box into global memory (completion: bulk group).
__device__ __forceinline__ void tma_reduce_add_3d(const CUtensorMap* map, const void* src, int x, int y,
                                                  int z) {
    asm volatile(
        "cp.reduce.async.bulk.tensor.3d.global.shared::cta.add.tile.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
            reinterpret_cast<uint64_t>(map)),
        "r"(smem_u32(src)), "r"(x), "r"(y), "r"(z)
        : "memory");
}

// a * b on bf16 pairs, rounded once (the product of two bf16 values is exact in fp32).
__device__ __forceinline__ uint32_t mul_bf16x2(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

// The low (h = 0) or high (h = 1) bf16 of w in both halves.
template <int h>
__device__ __forceinline__ uint32_t bcast_bf16(uint32_t w) {
    return h ? __byte_perm(w, 0u, 0x3232) : __byte_perm(w, 0u, 0x1010);
}


// One CTA: slices 2 grp and 2 grp + 1 of head bh (blockIdx = bh * groups + grp).
__global__ void __launch_bounds__(NT, 1)
poly_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
               const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmAcc,
               const PolyParams p) {
    constexpr uint32_t ID_O = idesc_bf16(128, NE, false, true);  // phi(Q) [S | Z], P [V | 1]
    constexpr uint32_t ID_S = idesc_bf16(128, NE, true, true);   // phi(K)^T [V | 1]
    constexpr uint32_t ID_P = idesc_bf16(128, 128, false, false);
    constexpr int G = plan::kPolyTcGroups;
    extern __shared__ __align__(1024) uint8_t sm[];
    const int t = threadIdx.x, warp = t >> 5;
    if (smem_u32(sm) & 1023u) {
        if (t == 0) atomicOr(p.status, kErrAlign);
        return;
    }
    uint64_t* tma_bar = reinterpret_cast<uint64_t*>(sm + Lay::BARS);  // the chunk's Q, K copies
    uint64_t* p_bar = tma_bar + 1;                                     // P = Q K^T
    uint64_t* a_bar = tma_bar + 2;  // a slice's products (the second: and P [V | 1])
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tma_bar + 3);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tma_bar + 4);
    uint64_t* v_bar = tma_bar + 5;  // the chunk's V copy
    if (t == 0) {
        mbar_init(tma_bar, 1);
        mbar_init(v_bar, 1);
        mbar_init(p_bar, 1);
        mbar_init(a_bar, 1);
        fence_mbar_init();
        *abort_flag = 0;
    }
    if (warp == 0) {
        tmem_alloc(tmem_slot, Lay::T_COLS);
        tmem_relinquish();
    }
    {   // row t of the constant and starting tiles: ones in EXT chunks 4-5, zero Z chunks,
        // zero columns 32 .. 63 of the padded Q and K, zero state terms
        const uint4 one4 = make_uint4(0x3F803F80u, 0x3F803F80u, 0x3F803F80u, 0x3F803F80u);
        const uint4 zero4 = make_uint4(0u, 0u, 0u, 0u);
        for (int c = 0; c < 8; ++c) {
            *reinterpret_cast<uint4*>(sm + ext_off(t, c)) = c == 4 || c == 5 ? one4 : zero4;
            *reinterpret_cast<uint4*>(sm + Lay::EXT2 + swz(t, c)) = zero4;
            *reinterpret_cast<uint4*>(sm + Lay::S0 + swz(t, c)) = zero4;
            *reinterpret_cast<uint4*>(sm + Lay::S1 + swz(t, c)) = zero4;
            *reinterpret_cast<uint4*>(sm + Lay::S0L + swz(t, c)) = zero4;
            *reinterpret_cast<uint4*>(sm + Lay::S1L + swz(t, c)) = zero4;
            if (c >= 4) {
                *reinterpret_cast<uint4*>(sm + Lay::QP + swz(t, c)) = zero4;
                *reinterpret_cast<uint4*>(sm + Lay::KP + swz(t, c)) = zero4;
            }
        }
    }
    fence_proxy_async();
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tm = *tmem_slot;
    const int bh = blockIdx.x / G, grp = blockIdx.x - bh * G;
    const uint32_t lane = static_cast<uint32_t>(32 * warp) << 16;
    const uint32_t sQP = smem_u32(sm + Lay::QP), sKP = smem_u32(sm + Lay::KP);
    const uint32_t sFQ = smem_u32(sm + Lay::FQ), sFK = smem_u32(sm + Lay::FK);
    const uint32_t sV = smem_u32(sm + Lay::V);
    // the hi and lo terms of [S_j | Z_j] (index 2 j + lo), with the leading-byte offsets to their
    // Z chunks; ones in EXT chunks 4 .. 5
    const uint32_t sS[4] = {smem_u32(sm + Lay::S0), smem_u32(sm + Lay::S0L), smem_u32(sm + Lay::S1),
                            smem_u32(sm + Lay::S1L)};
    const uint32_t lbo_s[4] = {Lay::EXT - Lay::S0, Lay::EXT + 96 - Lay::S0L, Lay::EXT + 32 - Lay::S1,
                               Lay::EXT2 - Lay::S1L};
    constexpr uint32_t LBO_V = Lay::EXT + 64 - Lay::V;
    const bool intra = p.causal && grp == 0;
    uint32_t p_phase = 0, a_phase = 0;
    uint32_t put = 0, got = 0, put_v = 0, got_v = 0;  // thread 0: copies issued and waited for

    auto fail = [&](unsigned code) {
        atomicOr(p.status, code);
        *abort_flag = 1;
    };
    // One thread polls the barrier; the others wait at the CTA barrier.
    auto wait_bar = [&](uint64_t* bar, uint32_t& phase) {
        if (t == 0 && !mbar_wait(bar, phase, kWaitLimit)) fail(kErrWait);
        __syncthreads();
        phase ^= 1u;
    };
    // Q and K go out as soon as every thread has read its rows of the chunk before, V once
    // the chunk before has taken its last product (thread 0 only).
    auto load_qk = [&](int c0, bool wq, bool wk) {
        ++put;
        mbar_arrive_expect_tx(tma_bar, (wq ? 8192u : 0u) + (wk ? 8192u : 0u));
        if (wq) tma_load_3d(sm + Lay::QR, &tmQ, tma_bar, 0, c0, bh);
        if (wk) tma_load_3d(sm + Lay::KR, &tmK, tma_bar, 0, c0, bh);
    };
    auto load_v = [&](int c0) {
        ++put_v;
        mbar_arrive_expect_tx(v_bar, kAtom);
        tma_load_3d(sm + Lay::V, &tmV, v_bar, 0, c0, bh);
    };
    // Row t of phi(X) for slice j of this CTA into the tile at `tile`: feature 32 al + b of
    // the slice is x_a x_b with a = 8 grp + 4 j + al (xa holds x_{8 grp} .. x_{8 grp + 7}).
    auto build = [&](uint8_t* tile, const uint32_t (&x2)[16], const uint32_t (&xa)[4], int j) {
#pragma unroll
        for (int al = 0; al < 4; ++al) {
            const uint32_t w = xa[2 * j + (al >> 1)];
            const uint32_t f = (al & 1) ? bcast_bf16<1>(w) : bcast_bf16<0>(w);
            uint32_t pk[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) pk[i] = mul_bf16x2(f, x2[i]);
            store_row32(tile, kAtom, t, 32 * al, pk);
        }
    };
    auto read_row = [&](uint32_t off, uint32_t (&x2)[16], uint32_t (&xa)[4]) {
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const uint4 u = *reinterpret_cast<const uint4*>(sm + off + swz64(t, c));
            x2[4 * c] = u.x;
            x2[4 * c + 1] = u.y;
            x2[4 * c + 2] = u.z;
            x2[4 * c + 3] = u.w;
        }
        const uint4 a = *reinterpret_cast<const uint4*>(sm + off + swz64(t, grp));
        xa[0] = a.x;
        xa[1] = a.y;
        xa[2] = a.z;
        xa[3] = a.w;
    };
    // S (row t = feature) and Z of slice j as hi and lo bf16 terms, for the next read-out.
    auto copy_slice = [&](int j) {
        {
            const uint32_t ts = tm + lane + (j ? Lay::T_S1 : Lay::T_S0);
#pragma unroll
            for (int j0 = 0; j0 < M; j0 += 32) {
                float v[32];
                tmem_ld32(ts + j0, v);
                uint32_t hi[16], lo[16];
#pragma unroll
                for (int u = 0; u < 16; ++u) {
                    hi[u] = pack_bf16(v[2 * u], v[2 * u + 1]);
                    lo[u] = pack_bf16(v[2 * u] - __uint_as_float(hi[u] << 16),
                                      v[2 * u + 1] - __uint_as_float(hi[u] & 0xFFFF0000u));
                }
                store_row32(sm + (j ? Lay::S1 : Lay::S0), kAtom, t, j0, hi);
                store_row32(sm + (j ? Lay::S1L : Lay::S0L), kAtom, t, j0, lo);
            }
            float z[16];
            tmem_ld16(ts + M, z);
            const uint32_t zh = pack_bf16(z[0], z[0]);
            const float zr = z[0] - __uint_as_float(zh << 16);
            const uint32_t zl = pack_bf16(zr, zr);
            const uint4 h4 = make_uint4(zh, zh, zh, zh), l4 = make_uint4(zl, zl, zl, zl);
            *reinterpret_cast<uint4*>(sm + ext_off(t, 2 * j)) = h4;
            *reinterpret_cast<uint4*>(sm + ext_off(t, 2 * j + 1)) = h4;
            uint8_t* const zlo = sm + (j ? Lay::EXT2 : Lay::EXT);  // lo term of Z: EXT 6-7, EXT2 0-1
            const int c0 = j ? 0 : 6;
            *reinterpret_cast<uint4*>(zlo + swz(t, c0)) = l4;
            *reinterpret_cast<uint4*>(zlo + swz(t, c0 + 1)) = l4;
        }
    };

    for (int pass = 0; pass < (p.causal ? 1 : 2); ++pass) {
        const bool do_state = p.causal || pass == 0;  // state updates
        const bool do_out = p.causal || pass == 1;    // read-outs
        const bool need_k = do_state || intra, need_v = do_state || intra;
        if (t == 0) {
            load_qk(0, do_out, need_k);
            if (need_v) load_v(0);
        }
        for (int c = 0; c < p.CH; ++c) {
            const int c0 = c * L;
            if (t == 0) {
                if (!mbar_wait(tma_bar, got & 1u, kWaitLimit)) fail(kErrWait);
                ++got;
                tma_store_wait_read();  // the previous rows, staged over the phi tiles, are read out
            }
            __syncthreads();
            uint32_t q2[16], qa[4], k2[16], ka[4];
            if (do_out) read_row(Lay::QR, q2, qa);
            if (need_k) read_row(Lay::KR, k2, ka);
            if (intra) {
                store_row32(sm + Lay::QP, kAtom, t, 0, q2);
                store_row32(sm + Lay::KP, kAtom, t, 0, k2);
            }
            if (do_out) build(sm + Lay::FQ, q2, qa, 0);
            if (do_state) build(sm + Lay::FK, k2, ka, 0);
            fence_proxy_async();
            fence_before_sync();
            __syncthreads();
            fence_after_sync();
            if (*abort_flag) goto cleanup;
            if (t == 0) {
                if (c + 1 < p.CH) load_qk(c0 + L, do_out, need_k);  // every row is read
                if (intra) {  // P = Q K^T over the 32 real columns
#pragma unroll
                    for (int k = 0; k < D / 16; ++k)
                        mma_bf16(tm + Lay::T_P, sdesc(sQP + 32 * k, 16, 1024), sdesc(sKP + 32 * k, 16, 1024),
                                 ID_P, k > 0 ? 1u : 0u);
                    mma_commit(p_bar);
                }
                if (do_out)
#pragma unroll
                    for (int k = 0; k < FS / 16; ++k) {
                        const uint64_t a = sdesc(sFQ + (k >> 2) * kAtom + 32 * (k & 3), 16, 1024);
                        mma_bf16(tm + Lay::T_O, a, sdesc(sS[0] + 2048 * k, lbo_s[0], 1024), ID_O, k > 0 ? 1u : 0u);
                        mma_bf16(tm + Lay::T_O, a, sdesc(sS[1] + 2048 * k, lbo_s[1], 1024), ID_O, 1u);
                    }
                if (need_v) {  // V lands under the products above
                    if (!mbar_wait(v_bar, got_v & 1u, kWaitLimit)) fail(kErrWait);
                    ++got_v;
                }
                if (do_state)
#pragma unroll
                    for (int k = 0; k < L / 16; ++k)
                        mma_bf16(tm + Lay::T_S0, sdesc(sFK + 2048 * k, kAtom, 1024),
                                 sdesc(sV + 2048 * k, LBO_V, 1024), ID_S, (c > 0 || k > 0) ? 1u : 0u);
                mma_commit(a_bar);
            }
            if (intra) {  // P squared, masked to j <= i, packed to bf16 pairs in place
                wait_bar(p_bar, p_phase);
                fence_after_sync();
#pragma unroll
                for (int jb = 0; jb < 2; ++jb) {
                    const int j0 = 64 * jb;
                    uint32_t pk[32];
                    if (j0 > 32 * warp + 31) {  // the whole warp's rows are before these keys
#pragma unroll
                        for (int u = 0; u < 32; ++u) pk[u] = 0u;
                    } else {
                        float v[64];
                        tmem_ld64(tm + lane + Lay::T_P + j0, v);
#pragma unroll
                        for (int u = 0; u < 32; ++u) {
                            const int j = j0 + 2 * u;
                            pk[u] = pack_bf16(j <= t ? v[2 * u] * v[2 * u] : 0.f,
                                              j + 1 <= t ? v[2 * u + 1] * v[2 * u + 1] : 0.f);
                        }
                    }
                    tmem_st32u(tm + lane + Lay::T_P + 32 * jb, pk);
                }
            }
            wait_bar(a_bar, a_phase);  // the first slice's products: the phi tiles are free
            fence_after_sync();
            if (do_out) build(sm + Lay::FQ, q2, qa, 1);
            if (do_state) build(sm + Lay::FK, k2, ka, 1);
            fence_proxy_async();
            fence_before_sync();
            __syncthreads();
            fence_after_sync();
            if (t == 0) {  // the second slice (its products touch none of the first slice's tiles)
                if (do_out)
#pragma unroll
                    for (int k = 0; k < FS / 16; ++k) {
                        const uint64_t a = sdesc(sFQ + (k >> 2) * kAtom + 32 * (k & 3), 16, 1024);
                        mma_bf16(tm + Lay::T_O, a, sdesc(sS[2] + 2048 * k, lbo_s[2], 1024), ID_O, 1u);
                        mma_bf16(tm + Lay::T_O, a, sdesc(sS[3] + 2048 * k, lbo_s[3], 1024), ID_O, 1u);
                    }
                if (do_state)
#pragma unroll
                    for (int k = 0; k < L / 16; ++k)
                        mma_bf16(tm + Lay::T_S1, sdesc(sFK + 2048 * k, kAtom, 1024),
                                 sdesc(sV + 2048 * k, LBO_V, 1024), ID_S, (c > 0 || k > 0) ? 1u : 0u);
                if (intra)  // O_ext += P [V | 1], P read from TMEM
#pragma unroll
                    for (int k = 0; k < L / 16; ++k)
                        mma_bf16_ts(tm + Lay::T_O, tm + Lay::T_P + 8 * k, sdesc(sV + 2048 * k, LBO_V, 1024),
                                    ID_O, 1u);
                mma_commit(a_bar);
            }
            if (p.causal) copy_slice(0);  // the first slice's state is final: copied under these products
            wait_bar(a_bar, a_phase);  // every product of the chunk: its input tiles are free
            fence_after_sync();
            if (t == 0 && need_v && c + 1 < p.CH) load_v(c0 + L);
            if (do_out) {  // the partial [numerator | normaliser] rows, added into the accumulator:
                           // columns 32b .. 32b + 31 in box b (box 2: the normaliser block, the
                           // columns past 80 fall outside the accumulator and are not added)
#pragma unroll
                for (int b = 0; b < 2; ++b) {
                    float v[32];
                    tmem_ld32(tm + lane + Lay::T_O + 32 * b, v);
#pragma unroll
                    for (int u = 0; u < 8; ++u)
                        *reinterpret_cast<float4*>(sm + Lay::STG + b * kAtom + swz(t, u)) =
                            make_float4(v[4 * u], v[4 * u + 1], v[4 * u + 2], v[4 * u + 3]);
                }
                float d[16];
                tmem_ld16(tm + lane + Lay::T_O + M, d);
#pragma unroll
                for (int u = 0; u < 4; ++u)
                    *reinterpret_cast<float4*>(sm + Lay::STG + 2 * kAtom + swz(t, u)) =
                        make_float4(d[4 * u], d[4 * u + 1], d[4 * u + 2], d[4 * u + 3]);
            }
            fence_proxy_async();
            fence_before_sync();
            __syncthreads();
            fence_after_sync();
            if (do_out && t == 0) {
#pragma unroll
                for (int b = 0; b < 3; ++b) tma_reduce_add_3d(&tmAcc, sm + Lay::STG + b * kAtom, 32 * b, c0, bh);
                tma_store_commit();
            }
            if (p.causal) copy_slice(1);  // while the reduce reads the staged rows out
        }
        if (!p.causal && pass == 0) {  // the totals, for the read-out pass
            copy_slice(0);
            copy_slice(1);
            fence_proxy_async();
            fence_before_sync();
            __syncthreads();
            fence_after_sync();
        }
    }

cleanup:
    if (t == 0) {  // copies and reductions still in flight land before the CTA leaves
        for (; got < put; ++got) mbar_wait(tma_bar, got & 1u, kWaitLimit);
        for (; got_v < put_v; ++got_v) mbar_wait(v_bar, got_v & 1u, kWaitLimit);
        tma_store_wait_all();
    }
    fence_before_sync();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tm, Lay::T_COLS);
}

// O = acc[:, :M] / acc[:, M] in bf16; one thread per 8 outputs of a row.
__global__ void poly_tc_divide(const float* __restrict__ acc, __nv_bfloat16* __restrict__ O, size_t rows) {
    const size_t i = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (i >= rows * (M / 8)) return;
    const size_t r = i / (M / 8);
    const int g8 = static_cast<int>(i % (M / 8));
    const float* a = acc + r * NE;
    const float inv = 1.f / a[M];
    const float4 x0 = *reinterpret_cast<const float4*>(a + 8 * g8);
    const float4 x1 = *reinterpret_cast<const float4*>(a + 8 * g8 + 4);
    *reinterpret_cast<uint4*>(O + r * M + 8 * g8) =
        make_uint4(pack_bf16(x0.x * inv, x0.y * inv), pack_bf16(x0.z * inv, x0.w * inv),
                   pack_bf16(x1.x * inv, x1.y * inv), pack_bf16(x1.z * inv, x1.w * inv));
}

}  // namespace tpoly

namespace {

// 3-D map over a [BH][N][C] tensor with a {box0, 128, 1} box.
cudaError_t make_map_box(CUtensorMap* m, const void* base, CUtensorMapDataType dt, int esz, int BH, int N,
                         int C, int box0, CUtensorMapSwizzle sw) {
    tcf::EncodeTiled enc = tcf::encoder();
    if (!enc) return cudaErrorNotSupported;
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(C), static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(BH)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(C) * esz, static_cast<cuuint64_t>(N) * C * esz};
    cuuint32_t box[3] = {static_cast<cuuint32_t>(box0), static_cast<cuuint32_t>(tcf::L), 1};
    cuuint32_t es[3] = {1, 1, 1};
    CUresult r = enc(m, dt, 3, const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

}  // namespace

cudaError_t poly2_forward_tc(const LaunchCtx& c, const __nv_bfloat16* Q, const __nv_bfloat16* K,
                             const __nv_bfloat16* V, __nv_bfloat16* O, int BH, int N, bool causal) {
    using namespace tpoly;
    const size_t bytes = plan::poly2_tc_scratch(BH, N);
    float* acc = nullptr;
    cudaError_t e = scratch_alloc(c, reinterpret_cast<void**>(&acc), bytes);
    if (e != cudaSuccess) return e;
    do {
        CUtensorMap mQ, mK, mV, mA;
        if ((e = make_map_box(&mQ, Q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, BH, N, D, D, CU_TENSOR_MAP_SWIZZLE_64B)) ||
            (e = make_map_box(&mK, K, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, BH, N, D, D, CU_TENSOR_MAP_SWIZZLE_64B)) ||
            (e = tcf::make_map(&mV, V, BH, N, M)) || (e = tcf::make_map_f32(&mA, acc, BH, N, NE)))
            break;
        if ((e = cudaMemsetAsync(acc, 0, bytes, c.stream)) != cudaSuccess) break;
        if ((e = cudaFuncSetAttribute(poly_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, Lay::BYTES)))
            break;
        const PolyParams p{N, BH, (N + tcf::L - 1) / tcf::L, causal ? 1 : 0, c.status_word};
        poly_tc_kernel<<<BH * plan::kPolyTcGroups, NT, Lay::BYTES, c.stream>>>(mQ, mK, mV, mA, p);
        const size_t rows = static_cast<size_t>(BH) * N, threads = rows * (M / 8);
        poly_tc_divide<<<static_cast<unsigned>((threads + 255) / 256), 256, 0, c.stream>>>(acc, O, rows);
        note_launch(2);
        e = cudaGetLastError();
    } while (false);
    scratch_free(c, acc);
    return e;
}

}  // namespace la
