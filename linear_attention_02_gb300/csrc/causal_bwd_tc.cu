// causal_bwd_tc.cu -- causal linear-attention backward on the 5th-generation
// tensor core, bf16 storage with D = M = 64.
//
// With qf = phi(Q), kf = phi(K), den_i = qf_i.Z_i, the quotient rule gives
//   gn_i = G_i / den_i,   gd_i = -(G_i . O_i) / den_i
// and the numerator gradients of "Transformers are RNNs" section 三（一）4
// (eqs. gq-gv: a prefix state for phi(Q), a suffix state for phi(K) and V)
// become, per chunk c of L = 128 tokens with g = [gn | gd 0...0] (an M + 16
// wide row, matching the ones block appended to V):
//   dP     = tril(g [V | 1]^T)                 (= gn_i.V_j + gd_i for j <= i)
//   dqf_c  = g [S | Z]_{c-1}^T + dP kf_c       (prefix state)
//   dV_c   = P^T gn + kf_c R_{c+1}             (suffix state R = sum qf g^T)
//   dkf_c  = dP^T qf_c + [V | 1] [R | r]_{c+1}^T
// and dQ = dqf * phi'(Q), dK = dkf * phi'(K) with phi' = min(phi, 1).
//
// Two kernels over the same work split as the forward (the chunks of all heads,
// head-major, cut into equal ranges, one per CTA; a range's pieces in
// successive heads are its segments):
//   prefix kernel -- the first piece's starting S, Z come from the forward's
//     nearest state checkpoint plus a short aggregate pass, or, without
//     checkpoints, from phase 1 / look-back as in the forward (later pieces
//     start a head from zero); then per chunk: den (from the forward, or from
//     P and qf.Z by MMA), gn, gd (written to scratch), [dP | dqf] by one MMA,
//     dqf += dP kf with dP read from TMEM, dQ out; the first piece's sum
//     qf^T g (its share of R) is published for the suffix kernel when earlier
//     units of its head exist;
//   suffix kernel -- walks its chunks in reverse; the last piece starts from
//     the shares of the later units of its head (all complete, the prefix
//     kernel has finished), earlier pieces from zero: P^T and dP^T by MMA,
//     masked and packed in TMEM, dV = P^T gn + kf R and dkf = dP^T qf +
//     [V | 1][R | r]^T with P^T, dP^T read from TMEM, R += qf^T g.
// Each CTA has eight compute warps (the epilogues), one MMA warp (every MMA,
// TMA copy and store) and three transform warps (the next chunk's Q and K into
// the free one of two buffers, phi there), handing work over through mbarriers
// and named barriers, so the MMAs no epilogue waits for run underneath them.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>

#include "la_launch.h"
#include "la_plan.h"
#include "tc_common.cuh"

namespace la {
namespace tcb {

using namespace la::tcf;

constexpr int D = 64, M = 64;
constexpr int NE = M + 16;
constexpr int W = D * M + D;           // words of a published (S | Z) or (R | r) state
constexpr uint32_t S_ATOM = D * 128;   // one atom column of a D-row state tile

// prefix-kernel shared memory.  An MN-major operand of D = 64 rows is read by
// an M = 128 MMA as two atoms (the second one's rows land in accumulator lanes
// nobody reads), so the atom after each Q and K buffer must be allocated.  The
// bf16 state [S | Z] sits right under V and the ones atom: read K-major, the
// 192 rows [V ; S] (K columns 0 .. 63) and [1 ; Z] (columns 64 .. 79) are one
// B operand, so dP = g [V | 1]^T and dqf = g [S | Z]^T are one N = 192 product.
struct LayF {
    static constexpr uint32_t Q0 = 0, Q1 = kAtom, K0 = 2 * kAtom, K1 = 3 * kAtom;  // two buffers each
    static constexpr uint32_t V = 4 * kAtom;
    static constexpr uint32_t S_LO = V + kAtom;          // S: D rows x M columns (one S atom)
    static constexpr uint32_t ONES = S_LO + S_ATOM;      // the ones atom
    static constexpr uint32_t S_HI = ONES + kAtom;       // Z (and 15 copies): D rows
    static constexpr uint32_t VS_K = ONES - V;           // K-atom stride of the [V ; S] operand
    static constexpr uint32_t G = S_HI + S_ATOM, O = G + kAtom;
    static constexpr uint32_t GH = O + kAtom;            // [gn | gd 0..0]: gn atom + extension atom
    static constexpr uint32_t P = GH + 2 * kAtom;        // the dQ staging tile
    static constexpr uint32_t XCH = P + kAtom;           // 2 x [2][128] fp32 partial row sums
    static constexpr uint32_t BARS = XCH + 2048;
    static constexpr uint32_t BYTES = BARS + 128;
    static constexpr uint32_t T_P = 0, T_DQ = 128, T_DEN = 192, T_S = 224, T_R = 304;
    static constexpr uint32_t T_COLS = 512;
};
static_assert(LayF::K1 + 2 * kAtom <= LayF::BYTES && LayF::Q1 + kAtom == LayF::K0, "padding atoms");
static_assert(LayF::S_HI - LayF::S_LO == LayF::VS_K && LayF::O == LayF::G + kAtom, "operand layout");
static_assert(LayF::G % 1024 == 0 && LayF::ONES % 1024 == 0 && LayF::S_HI % 1024 == 0, "alignment");
static_assert(LayF::T_DQ == LayF::T_P + 128, "dP and dqf are one accumulator block");

constexpr int kBT = 256;  // two warpgroups: warp w reads TMEM lanes 32 (w % 4) ..., and the
                          // two warps of a lane quarter split the columns of every row

// suffix-kernel shared memory (Q, read MN-major as two atoms, is followed by allocated atoms)
struct LayR {
    static constexpr uint32_t Q0 = 0, Q1 = kAtom, K0 = 2 * kAtom, K1 = 3 * kAtom;  // two buffers each
    static constexpr uint32_t V = 4 * kAtom, ONES = 5 * kAtom;
    static constexpr uint32_t GH = 6 * kAtom;
    static constexpr uint32_t P = 8 * kAtom;     // the dK staging tile
    static constexpr uint32_t DP = 9 * kAtom;    // the dV staging tile
    static constexpr uint32_t R = 10 * kAtom;    // [R | r 0..0] bf16, 2 atoms of D rows
    static constexpr uint32_t BARS = R + 2 * S_ATOM;
    static constexpr uint32_t BYTES = BARS + 128;
    static constexpr uint32_t T_P = 0, T_DP = 128, T_DV = 256, T_DK = 320, T_R = 384;
    static constexpr uint32_t T_COLS = 512;
};
static_assert(LayR::Q1 + kAtom == LayR::K0 && LayR::ONES == LayR::V + kAtom, "layout");

struct BwdParams {
    int N, BH, CH, per;   // tokens, heads, chunks per head, chunks per unit
    float* sagg;          // [units][W] last piece's (sum kf V^T | sum kf), pieces stopping mid-head
    float* ragg;          // [units][W] first piece's (sum qf gn^T | sum qf gd)
    unsigned* flags;      // [units]
    unsigned* ticket;
    float* gd;            // [BH][N]
    const float* den;     // [BH][N] the forward's normaliser per token, or null (recomputed)
    const float* ckpt;    // the forward's state checkpoints (see kCkptChunks), or null
    unsigned* status;
    int withhold;         // test hook: a unit that does not publish its aggregate (-1: none)
    unsigned spin_limit;  // flag polls before a look-back gives up
};

constexpr uint32_t ID_P = idesc_bf16(128, 128, false, false);     // K-major x K-major
constexpr uint32_t ID_PQ = idesc_bf16(128, 128 + D, false, false);  // [dP | dqf]
constexpr uint32_t ID_NE_MNMN = idesc_bf16(128, NE, true, true);  // state updates
constexpr uint32_t ID_16_KMN = idesc_bf16(128, 16, false, true);  // qf . [Z block]
constexpr uint32_t ID_D_KK = idesc_bf16(128, D, false, false);
constexpr uint32_t ID_D_KMN = idesc_bf16(128, D, false, true);
constexpr uint32_t ID_M_KMN = idesc_bf16(128, M, false, true);

// K-major descriptor for K step k of a tile whose 64-column atoms are `atom` bytes apart.
// The start address is the descriptor's low field (address / 16, shared memory below
// 256 KB), so a step is the tile's descriptor plus a constant: the MMA warp builds one
// descriptor per operand and adds, instead of building one per K step.
__device__ __forceinline__ uint64_t kmaj(uint32_t base, int k, uint32_t atom) {
    return sdesc(base, 16, 1024) + (((k >> 2) * atom + 32 * (k & 3)) >> 4);
}
// MN-major descriptor for K step k (16 rows) of a tile whose atoms are `lbo` bytes apart.
__device__ __forceinline__ uint64_t mnmaj(uint32_t base, int k, uint32_t lbo) {
    return sdesc(base, lbo, 1024) + 128u * static_cast<uint32_t>(k);
}

// Reads 32 bf16 values of `row` (16-byte chunks c0 .. c0 + 3) of a swizzled
// 128-row atom column into fp32 (a bf16 is the high half of an fp32).
__device__ __forceinline__ void read_row32(const uint8_t* tile, int row, int c0, float (&v)[32]) {
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        const uint4 u = *reinterpret_cast<const uint4*>(tile + swz(row, c0 + c));
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            v[8 * c + 2 * k] = __uint_as_float(w[k] << 16);
            v[8 * c + 2 * k + 1] = __uint_as_float(w[k] & 0xFFFF0000u);
        }
    }
}

// This warpgroup's 64 columns [64 g, 64 g + 64) of row i of a 128 x 128 fp32
// TMEM block, masked to j <= i and rounded to bf16 into a K-major tile (when
// STORE).  Returns the sum of the masked fp32 values.
template <bool STORE>
__device__ __forceinline__ float masked_half(uint32_t taddr, uint8_t* tile, int i, int q, int g) {
    const int j0 = 64 * g;
    uint32_t pk[32];
    float sum = 0.f;
    if (j0 > 32 * q + 31) {
#pragma unroll
        for (int u = 0; u < 32; ++u) pk[u] = 0u;
    } else {
        float v[64];
        tmem_ld64(taddr + j0, v);
#pragma unroll
        for (int u = 0; u < 32; ++u) {
            const int j = j0 + 2 * u;
            const float a = j <= i ? v[2 * u] : 0.f;
            const float b = j + 1 <= i ? v[2 * u + 1] : 0.f;
            sum += a + b;
            pk[u] = pack_bf16(a, b);
        }
    }
    if (STORE) {
        store_row32(tile, kAtom, i, j0, *reinterpret_cast<const uint32_t(*)[16]>(pk));
        store_row32(tile, kAtom, i, j0 + 32, *reinterpret_cast<const uint32_t(*)[16]>(pk + 16));
    }
    return sum;
}

// The same masking for the A operand of an MMA reading tensor memory: the
// warpgroup's 64 columns of row i are rounded to bf16 and packed in pairs back
// into the first 32 of those columns (each warp rewrites only its own lanes and
// only columns it has already read), so K step k of the product sits at column
// 8k + 32 (k >= 4).
__device__ __forceinline__ void masked_half_to_tmem(uint32_t taddr, int i, int q, int g) {
    const int j0 = 64 * g;
    uint32_t pk[32];
    if (j0 > 32 * q + 31) {
#pragma unroll
        for (int u = 0; u < 32; ++u) pk[u] = 0u;
    } else {
        float v[64];
        tmem_ld64(taddr + j0, v);
#pragma unroll
        for (int u = 0; u < 32; ++u) {
            const int j = j0 + 2 * u;
            pk[u] = pack_bf16(j <= i ? v[2 * u] : 0.f, j + 1 <= i ? v[2 * u + 1] : 0.f);
        }
    }
    tmem_st32u(taddr + j0, pk);
}
// Transposed form: row j of a TMEM block holding X^T (columns i), masked to
// i >= j and packed in place like masked_half_to_tmem.
__device__ __forceinline__ void masked_half_t_to_tmem(uint32_t taddr, int j, int q, int g) {
    const int i0 = 64 * g;
    uint32_t pk[32];
    if (i0 + 63 < 32 * q) {
#pragma unroll
        for (int u = 0; u < 32; ++u) pk[u] = 0u;
    } else {
        float v[64];
        tmem_ld64(taddr + i0, v);
#pragma unroll
        for (int u = 0; u < 32; ++u) {
            const int i = i0 + 2 * u;
            pk[u] = pack_bf16(i >= j ? v[2 * u] : 0.f, i + 1 >= j ? v[2 * u + 1] : 0.f);
        }
    }
    tmem_st32u(taddr + i0, pk);
}
// TMEM column of K step k of an A operand packed by masked_half_to_tmem.
__device__ __forceinline__ uint32_t packed_a_col(int k) { return 8 * k + (k >= 4 ? 32 : 0); }

// This warpgroup's 32 columns of a 64-column TMEM row -> bf16 tile row, times
// phi'(x) = min(phi, 1) taken from `phi_tile` when given.
__device__ __forceinline__ void tmem_half_to_tile(uint32_t taddr, uint8_t* tile, int row, int g,
                                                  const uint8_t* phi_tile) {
    float v[32];
    tmem_ld32(taddr + 32 * g, v);
    if (phi_tile) {
        float f[32];
        read_row32(phi_tile, row, 4 * g, f);
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] *= fminf(f[j], 1.f);
    }
    uint32_t pk[16];
#pragma unroll
    for (int u = 0; u < 16; ++u) pk[u] = pack_bf16(v[2 * u], v[2 * u + 1]);
    store_row32(tile, kAtom, row, 32 * g, pk);
}

// State row d: this warpgroup's 32 of the M columns (and, for g == 0, the 16
// extension columns) from TMEM -> bf16 state tile [D rows].
__device__ __forceinline__ void state_half_to_tile(uint32_t taddr, uint8_t* tile, int d, int g,
                                                   uint32_t hi_off = S_ATOM) {
    float v[32];
    tmem_ld32(taddr + 32 * g, v);
    uint32_t pk[16];
#pragma unroll
    for (int u = 0; u < 16; ++u) pk[u] = pack_bf16(v[2 * u], v[2 * u + 1]);
    store_row32(tile, S_ATOM, d, 32 * g, pk);
    if (g == 0) {
        float z[16];
        tmem_ld16(taddr + M, z);
        uint32_t zk[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) zk[u] = pack_bf16(z[2 * u], z[2 * u + 1]);
        *reinterpret_cast<uint4*>(tile + hi_off + swz(d, 0)) = make_uint4(zk[0], zk[1], zk[2], zk[3]);
        *reinterpret_cast<uint4*>(tile + hi_off + swz(d, 1)) = make_uint4(zk[4], zk[5], zk[6], zk[7]);
    }
}

// Writes this warpgroup's 32 values of a state row into TMEM and the bf16
// state tile; g == 0 also writes the extension columns (`ext`, then
// `ext_rest` fifteen times).
__device__ __forceinline__ void put_state_half(uint32_t taddr, uint8_t* tile, int d, int g,
                                               const float (&vals)[32], float ext, float ext_rest,
                                               uint32_t hi_off = S_ATOM) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        float v[16];
#pragma unroll
        for (int u = 0; u < 16; ++u) v[u] = vals[16 * h + u];
        tmem_st16(taddr + 32 * g + 16 * h, v);
        const int c = 4 * g + 2 * h;
        *reinterpret_cast<uint4*>(tile + swz(d, c)) =
            make_uint4(pack_bf16(v[0], v[1]), pack_bf16(v[2], v[3]), pack_bf16(v[4], v[5]),
                       pack_bf16(v[6], v[7]));
        *reinterpret_cast<uint4*>(tile + swz(d, c + 1)) =
            make_uint4(pack_bf16(v[8], v[9]), pack_bf16(v[10], v[11]), pack_bf16(v[12], v[13]),
                       pack_bf16(v[14], v[15]));
    }
    if (g == 0) {
        float e[16];
        e[0] = ext;
#pragma unroll
        for (int u = 1; u < 16; ++u) e[u] = ext_rest;
        tmem_st16(taddr + M, e);
        const uint32_t e0 = pack_bf16(ext, ext_rest), er = pack_bf16(ext_rest, ext_rest);
        *reinterpret_cast<uint4*>(tile + hi_off + swz(d, 0)) = make_uint4(e0, er, er, er);
        *reinterpret_cast<uint4*>(tile + hi_off + swz(d, 1)) = make_uint4(er, er, er, er);
    }
}

// Sum of the published [D*M | D] states sp0 <= sp < sp1 of a head: this
// warpgroup's 32 columns of row d into `row`; returns the summed extension
// word (meaningful for g == 0).
__device__ __forceinline__ float sum_states(const float* base, int sp0, int sp1, int d, int g,
                                            float (&row)[32]) {
#pragma unroll
    for (int e = 0; e < 32; ++e) row[e] = 0.f;
    float x0 = 0.f;
    for (int sp = sp0; sp < sp1; ++sp) {
        const float4* a =
            reinterpret_cast<const float4*>(base + static_cast<size_t>(sp) * W + d * M + 32 * g);
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const float4 x = __ldcg(a + u);
            row[4 * u] += x.x;
            row[4 * u + 1] += x.y;
            row[4 * u + 2] += x.z;
            row[4 * u + 3] += x.w;
        }
        if (g == 0) x0 += __ldcg(base + static_cast<size_t>(sp) * W + D * M + d);
    }
    return x0;
}

// Publishes this warpgroup's part of TMEM state row d as fp32 [D*M | D].
__device__ __forceinline__ void publish_half(uint32_t taddr, float* out, int d, int g) {
    float v[32];
    tmem_ld32(taddr + 32 * g, v);
#pragma unroll
    for (int u = 0; u < 8; ++u)
        reinterpret_cast<float4*>(out + d * M + 32 * g)[u] =
            make_float4(v[4 * u], v[4 * u + 1], v[4 * u + 2], v[4 * u + 3]);
    if (g == 0) {
        float z[16];
        tmem_ld16(taddr + M, z);
        out[D * M + d] = z[0];
    }
}

// CTA roles: warps 0 .. 7 compute (epilogues, one TMEM lane quarter and column
// half each), warp 8 issues every MMA, TMA copy and store (lane 0) and hands
// work to and from the compute warps, warps 9 .. 11 transform (load Q and K
// of the next chunk, apply phi; one on each scheduler the MMA warp leaves).  Because no compute thread issues MMAs, the
// MMAs that no epilogue waits for run underneath the epilogues.
constexpr int kMW = kBT / 32;             // the MMA warp
constexpr int kTW = 3;                    // transform warps
constexpr int kTT = 32 * kTW;             // their threads
constexpr int kT0 = kBT + 32;             // first transform thread
constexpr int kCT = kT0 + kTT;            // threads per CTA
constexpr int kEM = kBT + 32;             // compute warps + MMA warp
// Named barriers: compute warps among themselves; transform warps; compute ->
// MMA warp hand-overs (compute warps arrive, the MMA warp waits); MMA warp ->
// compute hand-overs (the MMA warp arrives, the compute warps wait).  Within a
// chunk every compute -> MMA hand-over has its own barrier (kBarEM, kBarEM2,
// kBarEM3), and the compute warps wait at kBarME once a chunk, which the MMA
// warp passes only after it has taken all of the previous chunk's hand-overs:
// so no side arrives at a barrier twice before the other has met the first
// arrival, whatever the (bounded, after a timeout short) mbarrier waits do.
constexpr uint32_t kBarE = 3, kBarT = 2, kBarEM = 1, kBarME = 4;
constexpr uint32_t kBarEM2 = 5;  // the second compute -> MMA warp hand-over of a chunk
constexpr uint32_t kBarEM3 = 6;  // the third

// Hand-over among the compute warps when they issue MMAs themselves (phase 1):
// their shared-memory writes become visible to the tensor core and TMA, and
// tcgen05 work is ordered around it.
__device__ __forceinline__ void sync_tc() {
    fence_proxy_async();
    fence_before_sync();
    bar_sync(kBarE, kBT);
    fence_after_sync();
}
// Compute warps -> MMA warp: their shared-memory and TMEM writes are done.
__device__ __forceinline__ void hand_to_mma(uint32_t id = kBarEM) {
    fence_proxy_async();
    fence_before_sync();
    bar_arrive(id, kEM);
}
__device__ __forceinline__ void take_from_compute(uint32_t id = kBarEM) {
    bar_sync(id, kEM);
    fence_after_sync();
}
// MMA warp -> compute warps: the tiles it waited for are in, the buffers free.
__device__ __forceinline__ void hand_to_compute() {
    fence_before_sync();
    bar_arrive(kBarME, kEM);
}
__device__ __forceinline__ void take_from_mma() {
    bar_sync(kBarME, kEM);
    fence_after_sync();
}

// Barriers and flags at the end of shared memory.
struct Bars {
    uint64_t tma, mma;   // copies of the MMA warp (and of phase 1); MMA completion
    uint64_t full[2];    // Q, K copies of buffer b landed
    uint64_t ready[2];   // phi(Q), phi(K) of buffer b are in place
    uint64_t freeb[2];   // the chunk using buffer b is done with it
    uint64_t rbar;       // completion of each chunk's last MMAs (R update included)
    uint64_t cb[4];      // suffix kernel: P^T, dP^T, dV, dK products of each chunk, one
                         // barrier per product so no waiter can fall two phases behind
    uint32_t tmem, pad;
    int unit, broken, pad2, pad3;
};
static_assert(sizeof(Bars) <= 128, "barrier block");

// One thread's bounded wait for the phase of `bar` with the given parity.  A
// timeout sets the error word and marks the CTA broken; from then on every wait
// is short and the kernel runs its hand-over protocol to the end with the
// remaining work unguarded, so no thread is left waiting at a named barrier.
__device__ __forceinline__ void poll(uint64_t* bar, uint32_t parity, Bars* bars, unsigned* status) {
    volatile int* broken = &bars->broken;
    if (!mbar_wait(bar, parity, *broken ? 64u : kWaitLimit)) {
        atomicOr(status, kErrWait);
        *broken = 1;
    }
}

// Transform warps: for each global chunk of the unit's range [start, end) in
// processing order (reversed for the suffix kernel), load Q and K into buffer
// (i & 1) once the chunk before it in that buffer has released it, apply phi
// (zeroing K's rows past the end of the head) and hand the pair over.
__device__ __forceinline__ void transform_chunks(const CUtensorMap* tmQ, const CUtensorMap* tmK,
                                                 uint8_t* q0, uint8_t* q1, uint8_t* k0, uint8_t* k1,
                                                 Bars* bars, int start, int end, int CH, int N,
                                                 bool reverse, unsigned* status) {
    const int tt = threadIdx.x - kT0;
    const volatile int* broken = &bars->broken;
    int pend[2] = {-1, -1};  // parity of a copy into buffer b not seen to land (thread tt == 0)
    for (int i = 0; i < end - start; ++i) {
        const int gc = reverse ? end - 1 - i : start + i;
        const int bh = gc / CH;
        const int c0 = (gc - bh * CH) * L;
        const int b = i & 1;
        const uint32_t u = static_cast<uint32_t>(i) >> 1;
        uint8_t* const tq = b ? q1 : q0;
        uint8_t* const tk = b ? k1 : k0;
        if (tt == 0) {
            if (i >= 2) poll(&bars->freeb[b], (u - 1) & 1u, bars, status);
            mbar_arrive_expect_tx(&bars->full[b], 2 * kAtom);
            tma_load_3d(tq, tmQ, &bars->full[b], 0, c0, bh);
            tma_load_3d(tk, tmK, &bars->full[b], 0, c0, bh);
            poll(&bars->full[b], u & 1u, bars, status);
            pend[b] = *broken ? static_cast<int>(u & 1u) : -1;
        }
        bar_sync(kBarT, kTT);
        const int valid = min(L, N - c0);
        phi_pair<kTT>(tq, tk, valid, tt);
        fence_proxy_async();
        bar_sync(kBarT, kTT);
        if (tt == 0) mbar_arrive(&bars->ready[b]);
    }
    if (tt == 0)  // copies not seen to land: wait for them before the CTA exits
        for (int b = 0; b < 2; ++b)
            if (pend[b] >= 0) mbar_wait(&bars->full[b], static_cast<uint32_t>(pend[b]), kWaitLimit);
}

// Bookkeeping of one thread's TMA loads on `tma`: how many phases it has
// opened, and the bytes expected on the open one but not issued yet, so that a
// kernel ending early can still drain the copies it started.
struct TmaBook {
    bool pending = false;
    uint32_t missing = 0;
    uint32_t count = 0;  // phases opened on the barrier so far (by any thread, in order)
    __device__ void expect(uint64_t* bar, uint32_t bytes) {
        mbar_arrive_expect_tx(bar, bytes);
        pending = true;
        missing = bytes;
        ++count;
    }
    __device__ void load(void* dst, const CUtensorMap* map, uint64_t* bar, int x, int y, int z) {
        tma_load_3d(dst, map, bar, x, y, z);
        missing -= kAtom;
    }
    __device__ void drain(uint64_t* bar) {
        if (!pending) return;
        if (missing) mbar_complete_tx(bar, missing);
        mbar_wait(bar, (count - 1) & 1u, kWaitLimit);
        pending = false;
    }
};

// ------------------------------------------------------------ prefix kernel

__global__ void __launch_bounds__(kCT, 1)
bwd_prefix_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                     const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmG,
                     const __grid_constant__ CUtensorMap tmO, const __grid_constant__ CUtensorMap tmGn,
                     const __grid_constant__ CUtensorMap tmdQ, const BwdParams p) {
    using Lay = LayF;
    extern __shared__ __align__(1024) uint8_t sm[];
    const int t = threadIdx.x, warp = t >> 5;
    const int q = warp & 3, g = (warp >> 2) & 1, row = 32 * q + (t & 31);
    if (smem_u32(sm) & 1023u) {
        if (t == 0) atomicOr(p.status, kErrAlign);
        return;
    }
    Bars* bars = reinterpret_cast<Bars*>(sm + Lay::BARS);
    uint64_t* tma_bar = &bars->tma;
    uint64_t* mma_bar = &bars->mma;
    float* xch = reinterpret_cast<float*>(sm + Lay::XCH);  // [2 sums][2 warpgroups][128 rows]
    if (t == 0) {
        mbar_init(tma_bar, 1);
        mbar_init(mma_bar, 1);
        mbar_init(&bars->rbar, 1);
        for (int b = 0; b < 2; ++b) {
            mbar_init(&bars->full[b], 1);
            mbar_init(&bars->ready[b], 1);
            mbar_init(&bars->freeb[b], 1);
        }
        fence_mbar_init();
        bars->broken = 0;
    }
    if (warp == 0) {
        tmem_alloc(&bars->tmem, Lay::T_COLS);
        tmem_relinquish();
    }
    for (int i = t; i < static_cast<int>(kAtom / 16); i += kCT)
        reinterpret_cast<uint4*>(sm + Lay::ONES)[i] =
            make_uint4(0x3F803F80u, 0x3F803F80u, 0x3F803F80u, 0x3F803F80u);
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tm = bars->tmem;
    if (t == 0) bars->unit = static_cast<int>(atomicAdd(p.ticket, 1u));
    __syncthreads();

    const int unit = bars->unit;
    const UnitRange ur(unit, p.per, p.CH, p.BH);
    const int first_end = min(ur.end, (ur.hA + 1) * p.CH);  // end of the first piece
    const bool have_den = p.den != nullptr;
    const int g0 = max(ur.start, ur.hB * p.CH);           // phase 1 covers [g0, end) when publishing
    // chunks of the aggregate pass before phase 2 (each opens one phase of the TMA and MMA
    // barriers): phase 1, or with checkpoints the way from the nearest one to the first piece
    const uint32_t n1 = static_cast<uint32_t>(
        p.ckpt ? (ur.look ? (ur.start - ur.hA * p.CH) % kCkptChunks : 0)
               : (ur.publish ? ur.end - g0 : 0));
    const uint32_t lane = static_cast<uint32_t>(32 * q) << 16;
    const uint32_t sV = smem_u32(sm + Lay::V), sGh = smem_u32(sm + Lay::GH);
    const uint32_t sSh = smem_u32(sm + Lay::S_HI);
    TmaBook book;  // thread 0 (phase 1) or the MMA warp's lane 0 (phase 2)

    // S_ext (+)= kf^T [V | 1] from K at sK and V at sv, its ones atom lbo bytes after it
    auto mma_state_update = [&](uint32_t sK, uint32_t sv, uint32_t lbo, bool accumulate_first) {
#pragma unroll
        for (int k = 0; k < L / 16; ++k)
            mma_bf16(tm + Lay::T_S, mnmaj(sK, k, kAtom), mnmaj(sv, k, lbo), ID_NE_MNMN,
                     (accumulate_first || k > 0) ? 1u : 0u);
    };

    // ------ phase 1 (aggregate of a last piece that stops mid-head) and look-back, compute warps
    // Phase 1 alternates K and V between (K0, V) and (K1, G) -- a ones atom written into O,
    // right after G -- so the next chunk's copy overlaps this chunk's phi and MMA.
    auto prelude = [&]() -> bool {  // false: give up
        uint32_t tma_phase = 0, mma_phase = 0;
        auto wait_bar = [&](uint64_t* bar, uint32_t& phase) -> bool {  // true: give up
            bool bad = false;
            if (t == 0 && !mbar_wait(bar, phase, kWaitLimit)) {
                atomicOr(p.status, kErrWait);
                bad = true;
            }
            phase ^= 1u;
            return bar_sync_or(kBarE, kBT, bad);
        };
        // T_S (+)= sum over the chunks [ga, gb) of head h of kf^T [V | 1]: onto its contents
        // when acc, from zero otherwise.
        auto aggregate = [&](int h, int ga, int gb, bool acc) -> bool {
            if (ga >= gb) return true;
            auto load_kv = [&](int c0, int b) {  // thread 0 only
                book.expect(tma_bar, 2 * kAtom);
                book.load(sm + (b ? Lay::K1 : Lay::K0), &tmK, tma_bar, 0, c0, h);
                book.load(sm + (b ? Lay::G : Lay::V), &tmV, tma_bar, 0, c0, h);
            };
            for (int i = t; i < static_cast<int>(kAtom / 16); i += kBT)
                reinterpret_cast<uint4*>(sm + Lay::O)[i] =
                    make_uint4(0x3F803F80u, 0x3F803F80u, 0x3F803F80u, 0x3F803F80u);
            fence_proxy_async();
            if (t == 0) load_kv((ga - h * p.CH) * L, 0);
            for (int gc = ga; gc < gb; ++gc) {
                const int c0 = (gc - h * p.CH) * L;
                const int b = (gc - ga) & 1;
                if (wait_bar(tma_bar, tma_phase)) return false;
                if (t == 0) book.pending = false;
                if (gc > ga) {  // the previous chunk's MMA has released the other buffer
                    if (wait_bar(mma_bar, mma_phase)) return false;
                    fence_after_sync();
                }
                if (t == 0 && gc + 1 < gb) load_kv(c0 + L, b ^ 1);
                phi_tile<true, kBT>(sm + (b ? Lay::K1 : Lay::K0), 1, min(L, p.N - c0));
                sync_tc();
                if (t == 0) {
                    mma_state_update(smem_u32(sm + (b ? Lay::K1 : Lay::K0)), b ? smem_u32(sm + Lay::G) : sV,
                                     b ? kAtom : Lay::VS_K, acc || gc > ga);
                    mma_commit(mma_bar);
                }
            }
            if (wait_bar(mma_bar, mma_phase)) return false;
            fence_after_sync();
            return true;
        };
        if (p.ckpt) {  // the first piece starts from the forward's nearest checkpoint
            float vals[32];
            float z = 0.f;
#pragma unroll
            for (int e = 0; e < 32; ++e) vals[e] = 0.f;
            const int h = ur.hA, kc = (ur.start - h * p.CH) / kCkptChunks;
            if (ur.look && kc > 0 && q < D / 32) {
                const float* ck = p.ckpt + (static_cast<size_t>(h) * ckpt_slots(p.CH) + kc) * W;
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const float4 x = __ldg(reinterpret_cast<const float4*>(ck + row * M + 32 * g) + u);
                    vals[4 * u] = x.x;
                    vals[4 * u + 1] = x.y;
                    vals[4 * u + 2] = x.z;
                    vals[4 * u + 3] = x.w;
                }
                z = __ldg(ck + D * M + row);
            }
            if (q < D / 32) put_state_half(tm + lane + Lay::T_S, sm + Lay::S_LO, row, g, vals, z, z, Lay::VS_K);
            sync_tc();
            if (ur.look) {  // the chunks between the checkpoint and the piece
                if (!aggregate(h, h * p.CH + kc * kCkptChunks, ur.start, true)) return false;
                if (q < D / 32) state_half_to_tile(tm + lane + Lay::T_S, sm + Lay::S_LO, row, g, Lay::VS_K);
                sync_tc();
            }
            return true;
        }
        if (ur.publish) {  // phase 1: the last piece's aggregate, for the later units of its head
            if (!aggregate(ur.hB, g0, ur.end, false)) return false;
            if (q < D / 32) publish_half(tm + lane + Lay::T_S, p.sagg + static_cast<size_t>(unit) * W, row, g);
            __threadfence();
            fence_before_sync();
            bar_sync(kBarE, kBT);
            if (t == 0 && unit != p.withhold) st_release(p.flags + unit, 1u);
        }
        bool bad = false;
        if (t == 0 && ur.look) {
            for (int sp = ur.u_first; sp < unit && !bad; ++sp) {
                uint32_t n = 0;
                while (ld_acquire(p.flags + sp) == 0u) {
                    if (++n > p.spin_limit) {
                        atomicOr(p.status, kErrLookback);
                        bad = true;
                        break;
                    }
                    __nanosleep(256);
                }
            }
        }
        if (bar_sync_or(kBarE, kBT, bad)) return false;
        if (q < D / 32) {
            float vals[32];
            const float z = sum_states(p.sagg, ur.look ? ur.u_first : unit, unit, row, g, vals);
            put_state_half(tm + lane + Lay::T_S, sm + Lay::S_LO, row, g, vals, z, z, Lay::VS_K);
        }
        sync_tc();
        return true;
    };
    const bool bad_pre = warp < kMW && !prelude();
    if (__syncthreads_or(bad_pre)) goto cleanup;

    // --------------------------------------------------- phase 2: dQ, gn, gd
    if (warp > kMW) {  // transform warps
        transform_chunks(&tmQ, &tmK, sm + Lay::Q0, sm + Lay::Q1, sm + Lay::K0, sm + Lay::K1, bars,
                         ur.start, ur.end, p.CH, p.N, false, p.status);
    } else if (warp == kMW) {  // MMA warp: lane 0 issues, the warp meets the hand-overs
        const bool lead = (t & 31) == 0;
        uint32_t tma_phase = n1 & 1u;  // phase 1 completed n1 phases of each barrier
        uint32_t ncommit = n1;         // commits to mma_bar so far
        uint32_t r_phase = 0;
        book.count = n1;
        if (lead) {  // V, G, O of the first chunk; Q and K come from the transform warps
            const int c0 = (ur.start - ur.hA * p.CH) * L;
            book.expect(tma_bar, 3 * kAtom);
            book.load(sm + Lay::V, &tmV, tma_bar, 0, c0, ur.hA);
            book.load(sm + Lay::G, &tmG, tma_bar, 0, c0, ur.hA);
            book.load(sm + Lay::O, &tmO, tma_bar, 0, c0, ur.hA);
        }
        for (int gc = ur.start; gc < ur.end; ++gc) {
            const int bh = gc / p.CH, c0 = (gc - bh * p.CH) * L;
            const int hn = (gc + 1) / p.CH, cn0 = (gc + 1 - hn * p.CH) * L;  // the next chunk
            const bool more = gc + 1 < ur.end;
            // qf^T g of the first piece is published for the earlier units of its head (none when
            // the piece starts the head)
            const bool in_first = ur.look && gc < first_end;
            const bool publish_here = ur.look && gc == first_end - 1;  // read out after this chunk
            const int b = (gc - ur.start) & 1;
            const uint32_t u = static_cast<uint32_t>(gc - ur.start) >> 1;
            const uint32_t sQ = smem_u32(sm + (b ? Lay::Q1 : Lay::Q0));
            const uint32_t sK = smem_u32(sm + (b ? Lay::K1 : Lay::K0));
            auto mma_r = [&]() {  // the first piece's share of R: qf^T g
#pragma unroll
                for (int k = 0; k < L / 16; ++k)
                    mma_bf16(tm + Lay::T_R, mnmaj(sQ, k, kAtom), mnmaj(sGh, k, kAtom), ID_NE_MNMN,
                             (gc > ur.start || k > 0) ? 1u : 0u);
            };
            if (lead) {
                poll(tma_bar, tma_phase, bars, p.status);  // V, G, O
                tma_phase ^= 1u;
                book.pending = false;
                if (more) book.expect(tma_bar, 3 * kAtom);
                if (gc > ur.start) {  // the previous chunk's MMAs are all done: its Q, K are free
                    poll(&bars->rbar, r_phase, bars, p.status);
                    r_phase ^= 1u;
                    mbar_arrive(&bars->freeb[b ^ 1]);
                }
                tma_store_wait_read_but_last();  // the g tile is read out (the dQ store may go on)
            }
            __syncwarp();
            hand_to_compute();  // G, O in; the g tile free: the compute warps start on gn, gd
            if (lead) {
                poll(&bars->ready[b], u & 1u, bars, p.status);  // phi(Q), phi(K)
                fence_after_sync();
                if (!have_den) {  // den = rowsum(tril(qf kf^T)) + qf . Z
#pragma unroll
                    for (int k = 0; k < D / 16; ++k) {
                        mma_bf16(tm + Lay::T_P, kmaj(sQ, k, kAtom), kmaj(sK, k, kAtom), ID_P, k > 0);
                        mma_bf16(tm + Lay::T_DEN, kmaj(sQ, k, kAtom), mnmaj(sSh, k, S_ATOM),
                                 ID_16_KMN, k > 0);
                    }
                    mma_commit(mma_bar);
                    ++ncommit;
                }
                mma_state_update(sK, sV, Lay::VS_K, true);  // S_c, read after the dP commit
            }
            __syncwarp();
            take_from_compute();  // the g tile (gn | gd) is written
            if (lead) {
                if (more) {  // G and O are consumed
                    book.load(sm + Lay::G, &tmG, tma_bar, 0, cn0, hn);
                    book.load(sm + Lay::O, &tmO, tma_bar, 0, cn0, hn);
                }
                tma_store_3d(&tmGn, sm + Lay::GH, 0, c0, bh);
                tma_store_commit();
#pragma unroll
                for (int k = 0; k < NE / 16; ++k)  // [dP | dqf] = g [V | 1 ; S | Z]^T
                    mma_bf16(tm + Lay::T_P, kmaj(sGh, k, kAtom), kmaj(sV, k, Lay::VS_K), ID_PQ, k > 0);
                mma_commit(mma_bar);
                const uint32_t dp_commit = ncommit++;
                if (publish_here) mma_r();  // covered by the next commit: read out after this chunk
                poll(mma_bar, dp_commit & 1u, bars, p.status);  // V is consumed (S update, dP)
                if (more) book.load(sm + Lay::V, &tmV, tma_bar, 0, cn0, hn);
            }
            __syncwarp();
            take_from_compute(kBarEM2);  // dP is masked and packed in TMEM
            if (lead) {
                tma_store_wait_read_but_last();  // the previous dQ store is read out: the staging
                                                 // tile is free once this chunk's MMA3 commits
#pragma unroll
                for (int k = 0; k < L / 16; ++k)  // dqf += dP kf, dP read from TMEM
                    mma_bf16_ts(tm + Lay::T_DQ, tm + Lay::T_P + packed_a_col(k), mnmaj(sK, k, kAtom),
                                ID_D_KMN, 1u);
                mma_commit(mma_bar);
                ++ncommit;
                if (in_first && !publish_here) mma_r();  // under the dQ epilogue
                mma_commit(&bars->rbar);
            }
            __syncwarp();
            take_from_compute(kBarEM3);  // dQ staged, S_c copied
            if (lead) {
                tma_store_3d(&tmdQ, sm + Lay::P, 0, c0, bh);
                tma_store_commit();
            }
        }
        if (lead) poll(&bars->rbar, r_phase, bars, p.status);  // the last chunk's MMAs
    } else {  // compute warps
        uint32_t e_commit = n1;  // commits to mma_bar waited for so far
        auto wait_mma = [&]() {
            if (t == 0) poll(mma_bar, e_commit & 1u, bars, p.status);
            ++e_commit;
            bar_sync(kBarE, kBT);
            fence_after_sync();
        };
        for (int gc = ur.start; gc < ur.end; ++gc) {
            const int bh = gc / p.CH, cc = gc - bh * p.CH;
            const int c0 = cc * L;
            const int valid = min(L, p.N - c0);
            const bool next_head = gc + 1 < ur.end && cc == p.CH - 1;  // the next chunk starts a head
            const int b = (gc - ur.start) & 1;
            uint8_t* const tQ = sm + (b ? Lay::Q1 : Lay::Q0);
            const float den_in =
                have_den && row < valid ? __ldg(p.den + static_cast<size_t>(bh) * p.N + c0 + row) : 1.f;
            take_from_mma();
            if (!have_den) wait_mma();
            {   // den, gn, gd -> g tile (bf16) and gd scratch
                const float part = have_den ? 0.f : masked_half<false>(tm + lane + Lay::T_P, nullptr, row, q, g);
                float gv[32], ov[32];
                read_row32(sm + Lay::G, row, 4 * g, gv);
                read_row32(sm + Lay::O, row, 4 * g, ov);
                float go = 0.f;
#pragma unroll
                for (int e = 0; e < 32; ++e) go = fmaf(gv[e], ov[e], go);
                xch[g * 128 + row] = part;
                xch[256 + g * 128 + row] = go;
                float dz0 = 0.f;
                if (!have_den) {
                    float dz[16];
                    tmem_ld16(tm + lane + Lay::T_DEN, dz);
                    dz0 = dz[0];
                }
                bar_sync(kBarE, kBT);
                const float den = have_den ? den_in : xch[row] + xch[128 + row] + dz0;
                const float go_all = xch[256 + row] + xch[384 + row];
                const bool ok = row < valid;
                const float inv = ok ? 1.f / den : 0.f;
                const float gd = -go_all * inv;
                uint32_t pk[16];
#pragma unroll
                for (int u2 = 0; u2 < 16; ++u2) pk[u2] = pack_bf16(gv[2 * u2] * inv, gv[2 * u2 + 1] * inv);
                store_row32(sm + Lay::GH, kAtom, row, 32 * g, pk);
                if (g == 0) {
                    *reinterpret_cast<uint4*>(sm + Lay::GH + kAtom + swz(row, 0)) =
                        make_uint4(pack_bf16(gd, 0.f), 0u, 0u, 0u);
                    *reinterpret_cast<uint4*>(sm + Lay::GH + kAtom + swz(row, 1)) =
                        make_uint4(0u, 0u, 0u, 0u);
                    if (ok) p.gd[static_cast<size_t>(bh) * p.N + c0 + row] = gd;
                }
            }
            hand_to_mma();
            wait_mma();  // dP (and the S update before it)
            masked_half_to_tmem(tm + lane + Lay::T_P, row, q, g);  // dP, masked, bf16 in TMEM
            hand_to_mma(kBarEM2);
            wait_mma();  // dqf complete
            if (q < D / 32) {
                if (ur.look && gc == first_end - 1)  // the first piece is complete: publish its R share
                    publish_half(tm + lane + Lay::T_R, p.ragg + static_cast<size_t>(unit) * W, row, g);
                if (next_head) {  // the next chunk starts a head: zero state
                    float zero[32];
#pragma unroll
                    for (int e = 0; e < 32; ++e) zero[e] = 0.f;
                    put_state_half(tm + lane + Lay::T_S, sm + Lay::S_LO, row, g, zero, 0.f, 0.f, Lay::VS_K);
                } else {
                    state_half_to_tile(tm + lane + Lay::T_S, sm + Lay::S_LO, row, g, Lay::VS_K);  // S_c, Z_c
                }
            }
            tmem_half_to_tile(tm + lane + Lay::T_DQ, sm + Lay::P, row, g, tQ);  // dQ
            hand_to_mma(kBarEM3);
        }
    }

cleanup:
    if (t == 0 || t == 32 * kMW) {  // phase 1's or the MMA warp's copies and stores
        book.drain(tma_bar);
        tma_store_wait_all();
    }
    fence_before_sync();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tm, Lay::T_COLS);
}

// ------------------------------------------------------------ suffix kernel

__global__ void __launch_bounds__(kCT, 1)
bwd_suffix_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                     const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmGn,
                     const __grid_constant__ CUtensorMap tmdK, const __grid_constant__ CUtensorMap tmdV,
                     const BwdParams p) {
    using Lay = LayR;
    extern __shared__ __align__(1024) uint8_t sm[];
    const int t = threadIdx.x, warp = t >> 5;
    const int q = warp & 3, g = (warp >> 2) & 1, row = 32 * q + (t & 31);
    if (smem_u32(sm) & 1023u) {
        if (t == 0) atomicOr(p.status, kErrAlign);
        return;
    }
    Bars* bars = reinterpret_cast<Bars*>(sm + Lay::BARS);
    uint64_t* tma_bar = &bars->tma;
    uint64_t* mma_bar = &bars->mma;
    if (t == 0) {
        mbar_init(tma_bar, 1);
        mbar_init(mma_bar, 1);
        mbar_init(&bars->rbar, 1);
        for (int j = 0; j < 4; ++j) mbar_init(&bars->cb[j], 1);
        for (int b = 0; b < 2; ++b) {
            mbar_init(&bars->full[b], 1);
            mbar_init(&bars->ready[b], 1);
            mbar_init(&bars->freeb[b], 1);
        }
        fence_mbar_init();
        bars->broken = 0;
    }
    if (warp == 0) {
        tmem_alloc(&bars->tmem, Lay::T_COLS);
        tmem_relinquish();
    }
    for (int i = t; i < static_cast<int>(kAtom / 16); i += kCT)
        reinterpret_cast<uint4*>(sm + Lay::ONES)[i] =
            make_uint4(0x3F803F80u, 0x3F803F80u, 0x3F803F80u, 0x3F803F80u);
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tm = bars->tmem;

    const int unit = blockIdx.x;
    const UnitRange ur(unit, p.per, p.CH, p.BH);
    const uint32_t lane = static_cast<uint32_t>(32 * q) << 16;
    const uint32_t sV = smem_u32(sm + Lay::V), sGh = smem_u32(sm + Lay::GH);
    const uint32_t sR = smem_u32(sm + Lay::R);
    TmaBook book;  // the MMA warp's lane 0

    if (warp < kMW) {
        if (q < D / 32) {  // R, r after the last piece: the first-piece shares of the later units
            float vals[32];
            const int sp0 = ur.publish ? unit + 1 : 0, sp1 = ur.publish ? ur.u_last + 1 : 0;
            const float r = sum_states(p.ragg, sp0, sp1, row, g, vals);
            put_state_half(tm + lane + Lay::T_R, sm + Lay::R, row, g, vals, r, 0.f);
        }
        fence_proxy_async();
        fence_before_sync();
    }
    __syncthreads();
    fence_after_sync();

    if (warp > kMW) {  // transform warps
        transform_chunks(&tmQ, &tmK, sm + Lay::Q0, sm + Lay::Q1, sm + Lay::K0, sm + Lay::K1, bars,
                         ur.start, ur.end, p.CH, p.N, true, p.status);
    } else if (warp == kMW) {  // MMA warp: lane 0 issues, the warp writes gd and meets the hand-overs
        const int ln = t & 31;
        const bool lead = ln == 0;
        uint32_t tma_phase = 0, r_phase = 0;
        // gd of rows 4 ln .. 4 ln + 3 of global chunk gc (zero past the end of its head)
        auto gd_rows = [&](int gc, float (&v)[4]) {
            const int h = gc / p.CH, c0 = (gc - h * p.CH) * L;
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                const int i = 4 * ln + r;
                v[r] = i < p.N - c0 ? __ldcg(p.gd + static_cast<size_t>(h) * p.N + c0 + i) : 0.f;
            }
        };
        float gdn[4];
        gd_rows(ur.end - 1, gdn);
        if (lead) {  // V and g of the first chunk; Q and K come from the transform warps
            const int c0 = (ur.end - 1 - ur.hB * p.CH) * L;
            book.expect(tma_bar, 2 * kAtom);
            book.load(sm + Lay::V, &tmV, tma_bar, 0, c0, ur.hB);
            book.load(sm + Lay::GH, &tmGn, tma_bar, 0, c0, ur.hB);
        }
        for (int gc = ur.end - 1; gc >= ur.start; --gc) {
            const int bh = gc / p.CH, cc = gc - bh * p.CH;
            const int c0 = cc * L;
            const bool more = gc > ur.start;
            const int hn = (gc - 1) / p.CH, cn0 = (gc - 1 - hn * p.CH) * L;  // the next chunk (if more)
            const int i = ur.end - 1 - gc;
            const int b = i & 1;
            const uint32_t u = static_cast<uint32_t>(i) >> 1;
            const uint32_t sQ = smem_u32(sm + (b ? Lay::Q1 : Lay::Q0));
            const uint32_t sK = smem_u32(sm + (b ? Lay::K1 : Lay::K0));
            // gd into the extension atom of the g tile (the previous chunk's MMAs are done)
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                const int rr = 4 * ln + r;
                *reinterpret_cast<uint4*>(sm + Lay::GH + kAtom + swz(rr, 0)) =
                    make_uint4(pack_bf16(gdn[r], 0.f), 0u, 0u, 0u);
                *reinterpret_cast<uint4*>(sm + Lay::GH + kAtom + swz(rr, 1)) = make_uint4(0u, 0u, 0u, 0u);
            }
            if (more) gd_rows(gc - 1, gdn);
            fence_proxy_async();
            __syncwarp();
            if (lead) {
                poll(&bars->ready[b], u & 1u, bars, p.status);  // phi(Q), phi(K)
                if (i > 0) mbar_arrive(&bars->freeb[b ^ 1]);  // the previous chunk's Q, K
                fence_after_sync();
#pragma unroll
                for (int k = 0; k < D / 16; ++k)  // P^T = kf qf^T (needs no V or g)
                    mma_bf16(tm + Lay::T_P, kmaj(sK, k, kAtom), kmaj(sQ, k, kAtom), ID_P, k > 0);
                mma_commit(&bars->cb[0]);
            }
            __syncwarp();
            hand_to_compute();
            if (lead) {
                poll(tma_bar, tma_phase, bars, p.status);  // V, gn
                tma_phase ^= 1u;
                book.pending = false;
                if (more) book.expect(tma_bar, 2 * kAtom);
#pragma unroll
                for (int k = 0; k < NE / 16; ++k)  // dP^T = [V | 1] g^T
                    mma_bf16(tm + Lay::T_DP, kmaj(sV, k, kAtom), kmaj(sGh, k, kAtom), ID_P, k > 0);
                mma_commit(&bars->cb[1]);
            }
            __syncwarp();
            take_from_compute();  // P^T is masked and packed in TMEM
            if (lead) {
                tma_store_wait_read();  // the staging tiles are read out before dV, dK commit
#pragma unroll
                for (int k = 0; k < L / 16; ++k)  // dV = P^T gn, P^T read from TMEM
                    mma_bf16_ts(tm + Lay::T_DV, tm + Lay::T_P + packed_a_col(k), mnmaj(sGh, k, kAtom),
                                ID_M_KMN, k > 0);
#pragma unroll
                for (int k = 0; k < D / 16; ++k)  // dV += kf R
                    mma_bf16(tm + Lay::T_DV, kmaj(sK, k, kAtom), mnmaj(sR, k, S_ATOM), ID_M_KMN, 1u);
                mma_commit(&bars->cb[2]);
            }
            __syncwarp();
            take_from_compute(kBarEM2);  // dP^T is masked and packed in TMEM
            if (lead) {
#pragma unroll
                for (int k = 0; k < L / 16; ++k)  // dkf = dP^T qf, dP^T read from TMEM
                    mma_bf16_ts(tm + Lay::T_DK, tm + Lay::T_DP + packed_a_col(k), mnmaj(sQ, k, kAtom),
                                ID_D_KMN, k > 0);
#pragma unroll
                for (int k = 0; k < NE / 16; ++k)  // dkf += [V | 1] [R | r]^T
                    mma_bf16(tm + Lay::T_DK, kmaj(sV, k, kAtom), kmaj(sR, k, S_ATOM), ID_D_KK, 1u);
                mma_commit(&bars->cb[3]);
                if (cc > 0) {  // R += qf^T g (not needed before a head's first chunk)
#pragma unroll
                    for (int k = 0; k < L / 16; ++k)
                        mma_bf16(tm + Lay::T_R, mnmaj(sQ, k, kAtom), mnmaj(sGh, k, kAtom), ID_NE_MNMN, 1u);
                }
                mma_commit(&bars->rbar);
                poll(&bars->rbar, r_phase, bars, p.status);  // V and g are consumed
                r_phase ^= 1u;
                if (more) {
                    book.load(sm + Lay::V, &tmV, tma_bar, 0, cn0, hn);
                    book.load(sm + Lay::GH, &tmGn, tma_bar, 0, cn0, hn);
                }
            }
            __syncwarp();
            take_from_compute(kBarEM3);  // dK, dV staged, R_c copied
            if (lead) {
                tma_store_3d(&tmdK, sm + Lay::P, 0, c0, bh);
                tma_store_3d(&tmdV, sm + Lay::DP, 0, c0, bh);
                tma_store_commit();
            }
        }
    } else {  // compute warps
        uint32_t e_r = 0;
        auto wait_on = [&](uint64_t* bar, uint32_t parity) {
            if (t == 0) poll(bar, parity, bars, p.status);
            bar_sync(kBarE, kBT);
            fence_after_sync();
        };
        for (int gc = ur.end - 1; gc >= ur.start; --gc) {
            const int bh = gc / p.CH, cc = gc - bh * p.CH;
            const bool more = gc > ur.start;
            const int b = (ur.end - 1 - gc) & 1;
            const uint32_t ph = static_cast<uint32_t>(ur.end - 1 - gc) & 1u;  // this chunk's phase
            uint8_t* const tK = sm + (b ? Lay::K1 : Lay::K0);
            (void)bh;
            take_from_mma();
            wait_on(&bars->cb[0], ph);  // P^T
            masked_half_t_to_tmem(tm + lane + Lay::T_P, row, q, g);   // P^T, masked, bf16 in TMEM
            hand_to_mma();              // the dV products start
            wait_on(&bars->cb[1], ph);  // dP^T
            masked_half_t_to_tmem(tm + lane + Lay::T_DP, row, q, g);  // dP^T likewise
            hand_to_mma(kBarEM2);       // the dK products start
            wait_on(&bars->cb[2], ph);  // dV
            tmem_half_to_tile(tm + lane + Lay::T_DV, sm + Lay::DP, row, g, nullptr);  // dV
            wait_on(&bars->cb[3], ph);  // dkf
            tmem_half_to_tile(tm + lane + Lay::T_DK, sm + Lay::P, row, g, tK);        // dK
            wait_on(&bars->rbar, e_r & 1u);  // R_c
            ++e_r;
            if (q < D / 32) {
                if (cc > 0) {
                    state_half_to_tile(tm + lane + Lay::T_R, sm + Lay::R, row, g);  // R_c
                } else if (more) {  // the next chunk ends the previous head: R starts from zero
                    float zero[32];
#pragma unroll
                    for (int e = 0; e < 32; ++e) zero[e] = 0.f;
                    put_state_half(tm + lane + Lay::T_R, sm + Lay::R, row, g, zero, 0.f, 0.f);
                }
            }
            hand_to_mma(kBarEM3);
        }
    }

    if (t == 32 * kMW) {  // the MMA warp's copies and stores
        book.drain(tma_bar);
        tma_store_wait_all();
    }
    fence_before_sync();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tm, Lay::T_COLS);
}

}  // namespace tcb

size_t causal_backward_tc64_scratch(int BH, int N, int num_sms, bool out_given, bool den_given,
                                    bool ckpt_given) {
    using namespace tcb;
    static_assert(LayF::T_COLS == 512, "one CTA per SM");
    const int chunks = (N + L - 1) / L;
    const size_t units = static_cast<size_t>(plan::tc_units(BH, chunks, num_sms));
    const size_t agg = sizeof(float) * units * W, flags = sizeof(unsigned) * (units + 1);
    const size_t gn = sizeof(__nv_bfloat16) * static_cast<size_t>(BH) * N * M;
    const size_t gd = sizeof(float) * static_cast<size_t>(BH) * N;
    using plan::up256;
    size_t total = 2 * up256(agg) + up256(flags) + up256(gn) + up256(gd);
    if (!out_given) {  // Out recomputed: its tile, its normaliser, its checkpoints and the
                       // forward's own scratch, live at the same time
        total += up256(gn) + up256(gd);
        if (!ckpt_given) total += up256(sizeof(float) * static_cast<size_t>(BH) * ckpt_slots(chunks) * W);
        total += causal_forward_tc_scratch(64, BH, N, num_sms);
    }
    (void)den_given;  // the layout reserves the normaliser whenever Out is recomputed
    return total;
}

cudaError_t causal_backward_tc64(const LaunchCtx& c, const __nv_bfloat16* Q, const __nv_bfloat16* K,
                                 const __nv_bfloat16* V, const __nv_bfloat16* O,
                                 const __nv_bfloat16* G, __nv_bfloat16* dQ, __nv_bfloat16* dK,
                                 __nv_bfloat16* dV, int BH, int N, const float* Den,
                                 const float* Ckpt) {
    using namespace tcb;
    auto kf = bwd_prefix_tc_kernel;
    auto kr = bwd_suffix_tc_kernel;
    cudaError_t e;
    if ((e = cudaFuncSetAttribute(kf, cudaFuncAttributeMaxDynamicSharedMemorySize, LayF::BYTES)) ||
        (e = cudaFuncSetAttribute(kr, cudaFuncAttributeMaxDynamicSharedMemorySize, LayR::BYTES)) ||
        (e = cudaFuncSetAttribute(kf, cudaFuncAttributePreferredSharedMemoryCarveout,
                                  cudaSharedmemCarveoutMaxShared)) ||
        (e = cudaFuncSetAttribute(kr, cudaFuncAttributePreferredSharedMemoryCarveout,
                                  cudaSharedmemCarveoutMaxShared)))
        return e;
    int per_sm = 0;
    if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kf, kCT, LayF::BYTES)))
        return e;
    if (per_sm < 1) return cudaErrorInvalidConfiguration;
    const int chunks = (N + L - 1) / L;
    const int slots = c.num_sms;  // one CTA per SM (512 TMEM columns each)
    const ChunkSplit split = split_chunks(BH, chunks, slots);
    const int units = split.units;

    const size_t agg_bytes = sizeof(float) * static_cast<size_t>(units) * W;
    const size_t flag_bytes = sizeof(unsigned) * (static_cast<size_t>(units) + 1);
    const size_t gn_bytes = sizeof(__nv_bfloat16) * static_cast<size_t>(BH) * N * M;
    const size_t gd_bytes = sizeof(float) * static_cast<size_t>(BH) * N;
    const size_t o_bytes = O ? 0 : gn_bytes;
    const size_t den_bytes = O ? 0 : gd_bytes;  // the recomputed forward's normaliser
    const size_t ck_bytes =  // and its checkpoints
        O || Ckpt ? 0 : sizeof(float) * static_cast<size_t>(BH) * ckpt_slots(chunks) * W;
    auto up = [](size_t x) { return (x + 255) & ~static_cast<size_t>(255); };
    const size_t total = 2 * up(agg_bytes) + up(flag_bytes) + up(gn_bytes) + up(gd_bytes) + up(o_bytes) +
                         up(den_bytes) + up(ck_bytes);
    char* ws = nullptr;
    if (total != causal_backward_tc64_scratch(BH, N, c.num_sms, O != nullptr, Den != nullptr,
                                              Ckpt != nullptr) -
                     (O ? 0 : causal_forward_tc_scratch(64, BH, N, c.num_sms)))
        return cudaErrorInvalidValue;  // the plan and this layout must agree
    if ((e = scratch_alloc(c, reinterpret_cast<void**>(&ws), total)) != cudaSuccess) return e;
    BwdParams p;
    p.N = N;
    p.BH = BH;
    p.CH = chunks;
    p.per = split.per;
    char* q = ws;
    p.sagg = reinterpret_cast<float*>(q);
    q += up(agg_bytes);
    p.ragg = reinterpret_cast<float*>(q);
    q += up(agg_bytes);
    p.flags = reinterpret_cast<unsigned*>(q);
    p.ticket = p.flags + units;
    q += up(flag_bytes);
    __nv_bfloat16* gn = reinterpret_cast<__nv_bfloat16*>(q);
    q += up(gn_bytes);
    p.gd = reinterpret_cast<float*>(q);
    q += up(gd_bytes);
    __nv_bfloat16* Ow = O ? nullptr : reinterpret_cast<__nv_bfloat16*>(q);
    q += up(o_bytes);
    float* Dw = O ? nullptr : reinterpret_cast<float*>(q);
    q += up(den_bytes);
    float* Cw = ck_bytes ? reinterpret_cast<float*>(q) : nullptr;
    p.den = Den;
    p.ckpt = Ckpt;
    p.withhold = c.withhold_unit;
    p.spin_limit = c.spin_limit ? c.spin_limit : kSpinLimit;
    p.status = c.status_word;
    do {
        if (!O) {  // the output is needed for gd: recompute it
            if ((e = causal_forward_tc<64, 64>(c, Q, K, V, Ow, BH, N, nullptr, nullptr, nullptr,
                                               nullptr, Den ? nullptr : Dw, Cw)) != cudaSuccess)
                break;
            O = Ow;
            if (!Den) p.den = Dw;
            if (!Ckpt) p.ckpt = Cw;
        }
        if ((e = cudaMemsetAsync(p.flags, 0, flag_bytes, c.stream)) != cudaSuccess) break;
        CUtensorMap mQ, mK, mV, mG, mO, mGn, mdQ, mdK, mdV;
        if ((e = make_map(&mQ, Q, BH, N, D)) || (e = make_map(&mK, K, BH, N, D)) ||
            (e = make_map(&mV, V, BH, N, M)) || (e = make_map(&mG, G, BH, N, M)) ||
            (e = make_map(&mO, O, BH, N, M)) || (e = make_map(&mGn, gn, BH, N, M)) ||
            (e = make_map(&mdQ, dQ, BH, N, D)) || (e = make_map(&mdK, dK, BH, N, D)) ||
            (e = make_map(&mdV, dV, BH, N, M)))
            break;
        kf<<<units, kCT, LayF::BYTES, c.stream>>>(mQ, mK, mV, mG, mO, mGn, mdQ, p);
        kr<<<units, kCT, LayR::BYTES, c.stream>>>(mQ, mK, mV, mGn, mdK, mdV, p);
        note_launch(2);
        e = cudaGetLastError();
    } while (0);
    scratch_free(c, ws);
    return e;
}

}  // namespace la
