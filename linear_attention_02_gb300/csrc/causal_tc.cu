// causal_tc.cu -- chunked causal linear-attention forward on the 5th-generation
// tensor core (bf16 storage, fp32 accumulation), D = M in {64, 128}.
//
// The sequence of every head is cut into chunks of L = 128 tokens.  With phi(x) = elu(x) + 1 ("Transformers are RNNs",
// section 特征映射) applied in shared memory, a chunk c needs
//   P      = tril(phi(Q_c) phi(K_c)^T)                (intra-chunk scores, eq. mask)
//   O_ext  = phi(Q_c) [S | Z]_{c-1} + P [V_c | 1]     (numerator and normaliser)
//   S_ext += phi(K_c)^T [V_c | 1]                     (S_c and Z_c, the incremental update)
// and V'_c = O_ext[:, :M] / O_ext[:, M] (eq. output).  Appending a block of
// ones to V turns the normaliser sum phi(Q_i).Z_i into one more output column
// of the same products, so numerator and denominator see the same rounding of
// P and of the state.
//
// All four products run on tcgen05.mma (M = 128) with accumulators in TMEM:
//   P     [128 x 128]  A = phi(Q_c) K-major,  B = phi(K_c) K-major
//   S_ext [128 x NE]   A = phi(K_c)^T MN-major (D = 64 pads to 128 rows whose
//                      extra rows are never read), B = [V_c | 1] MN-major
//   O_ext [128 x NE]   A = phi(Q_c) K-major, B = [S | Z] (bf16 copy) MN-major
//                      then A = P (bf16, masked, packed in place in TMEM),
//                      B = [V_c | 1] MN-major
// Tiles arrive by TMA with the 128-byte swizzle; the bf16 state and the
// output tile are written by the threads in the same swizzled layout.
//
// Work split: the chunks of all heads, head-major, are cut into equal ranges,
// one per resident CTA, so a range may end inside a head and the next range
// continue it.  Phase 1 of a unit whose range stops inside a head accumulates
// that last piece's aggregate (sum phi(K)^T V | sum phi(K)) and publishes it
// with a release flag (1).  Phase 2 starts its first piece from the sum of the
// earlier aggregates of that head (bounded waits on their flags, walking
// back), and runs the chunk loop,
// restarting the state at every head boundary.  Units are taken from an atomic ticket after TMEM is
// allocated, so a CTA only ever waits for CTAs that started (and hold their
// TMEM) before it.  With very many ranges per head (D = 64) the walk is cut short:
// a piece that starts at its head's start also publishes the head's state at
// its end (flag 2), and so does every unit once its look-back is done; the
// walk stops at the first flag 2 it meets, and no unit ever waits for a
// state, only for aggregates.
//
// The same kernel, instantiated with RET, runs linear attention with decay
// ("retention", "Transformer and Variants" sections 1.3.2 and 1.3.4):
// S_t = gamma_t S_{t-1} + k_t v_t^T, y_t = S_t^T q_t, raw q and k, no
// normaliser.  With a_i the running sum of log2(gamma) over the chunk's tokens
// 0 .. i and A = a_127:
//   y_c   = (tril(Q_c K_c^T) * 2^(a_i - a_j)) V_c + diag(2^a) Q_c S_{c-1}
//   S_c   = 2^A S_{c-1} + (diag(2^(A - a)) K_c)^T V_c
// so P is scaled as it is masked, the Q and K tiles are scaled by rows after
// P is taken, and the fp32 state in TMEM is scaled before the update; every
// power of two has a non-positive exponent.  A published piece carries its
// total log2 decay, and the look-back decays each earlier aggregate by the
// pieces after it.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <mutex>

#include "la_launch.h"
#include "la_plan.h"
#include "tc_common.cuh"

namespace la {
namespace tcf {

template <int D, int M, bool RET = false>
struct Layout {
    static constexpr int DA = D / 64;  // atom columns of a phi(Q)/phi(K) tile
    static constexpr int MA = M / 64;  // atom columns of a V / output tile
    static constexpr int NE = M + 16;  // M values + 16 copies of the normaliser column
    static constexpr int W = D * M + D;  // words of a published (S | Z) state
    // D = 64: one warpgroup and 112 KB, so two CTAs share an SM and overlap each
    // other's waits; D = 128: one CTA per SM whose two warpgroups split the
    // element-wise work by columns (both measured faster than the alternatives).
    static constexpr int GROUPS = D == 64 ? 1 : 2;
    static constexpr int THREADS = 128 * GROUPS;
    // shared memory (byte offsets from a 1024-aligned base)
    static constexpr uint32_t Q = 0;
    static constexpr uint32_t K = Q + DA * kAtom;
    static constexpr uint32_t V = K + DA * kAtom;      // V atoms, then the ones atom
    static constexpr uint32_t ONES = V + MA * kAtom;
    static constexpr uint32_t P = ONES + kAtom;        // 2 atoms: the output staging tile (MA atoms),
                                                       // and phase 1's K, V buffers
    static constexpr uint32_t S = P + 2 * kAtom;       // (MA + 1) atoms of D rows
    static constexpr uint32_t S_ATOM = D * 128;
    // phase 1's third K, V buffer: the second P atom and the S tile (D = 64), the S tile and
    // 16 KB after it (D = 128)
    static constexpr uint32_t KV2_K = D == 64 ? P + kAtom : S;
    static constexpr uint32_t KV2_V = D == 64 ? S : S + DA * kAtom;
    static constexpr uint32_t BARS = S + (MA + 1) * S_ATOM > KV2_V + MA * kAtom ? S + (MA + 1) * S_ATOM
                                                                                 : KV2_V + MA * kAtom;
    static constexpr uint32_t DEC = BARS + 64;  // retention: a_i of the chunk (128 floats), warp sums
    static constexpr uint32_t BYTES = BARS + 64 + (RET ? 528 : 0);
    // tensor memory columns: P (fp32, then masked and packed in place to bf16 pairs, the A
    // operand of P [V | 1]: columns 0 .. 63 for one warpgroup, 0 .. 31 and 64 .. 95 for two),
    // O_ext after the packed P, S_ext after O_ext
    static constexpr uint32_t T_P = 0;
    static constexpr uint32_t T_O = GROUPS == 1 ? 64 : 128;
    static constexpr uint32_t T_S = T_O + NE;
    static constexpr uint32_t T_COLS = T_S + NE <= 256 ? 256 : 512;
    // packed column of K step k (16 keys) of P
    static __device__ __forceinline__ uint32_t p_col(int k) { return GROUPS == 1 ? 8 * k : 8 * k + (k >= 4 ? 32 : 0); }
    static constexpr uint32_t TX_QKV = (2 * DA + MA) * kAtom;
    static constexpr uint32_t TX_KV = (DA + MA) * kAtom;
    // CTAs that fit on one SM: 228 KB of shared memory (1 KB reserved per CTA)
    // and 512 TMEM columns.
    static constexpr int SMEM_FIT = static_cast<int>(233472u / (BYTES + 1024u));
    static constexpr int TMEM_FIT = static_cast<int>(512u / T_COLS);
    static constexpr int PER_SM = SMEM_FIT < TMEM_FIT ? SMEM_FIT : TMEM_FIT;
    static_assert(D == M && (D == 64 || D == 128), "tensor-core path covers D = M in {64, 128}");
    static_assert(BYTES <= 227 * 1024, "shared memory");
    static_assert(PER_SM >= 1, "one CTA must fit");
};

struct FwdParams {
    int N, BH, CH, per;    // tokens, heads, chunks per head, chunks per unit
    float* agg;            // [units][W] aggregate of each published piece
    float* incl;           // [units][W] the head's state at the end of each published piece
    int use_incl;          // publish and use those states (over 128 ranges per head, D = 64)
    unsigned* flags;       // [units], zero before the launch: 1 = aggregate published,
                           // 2 = inclusive state published as well
    unsigned* ticket;      // zero before the launch
    const float* S_init;   // [BH][D][M] or null
    const float* Z_init;   // [BH][D] or null
    float* S_final;        // [BH][D][M] or null
    float* Z_final;        // [BH][D] or null
    float* den;            // [BH][N] or null: the normaliser of every token
    float* ckpt;           // [BH][ckpt_slots(CH)][W] or null: states before every 8th chunk
    unsigned* status;      // device error word
    // retention only
    const float* gates;       // [BH][N] per-token decays, or null
    const float* gamma_head;  // [H] per-head decays, or null (neither: decay 1)
    int H;                    // heads per batch entry
    float* lam;               // [units] total log2 decay of each published piece
    int withhold;             // test hook: a unit that does not publish (-1: none)
    unsigned spin_limit;      // flag polls before a look-back gives up
};

// log2 of a decay, kept finite: a decay below 2^-64 counts as 2^-64.
__device__ __forceinline__ float log2_decay(float g) { return fmaxf(log2f(g), -64.f); }

// A chunk whose total log2 decay A is at least this has its decays factored into its rows:
// Q row i times 2^(a_i), K row j times 2^(-a_j) <= 2^100 (inside the range of bf16), so that
// P = Q K^T comes out as P_ij 2^(a_i - a_j) and the update S += K^T [V | 1] is scaled by 2^A
// afterwards.  A chunk with a stronger decay takes P's decay element by element.
constexpr float kFactorMin = -100.f;

// This thread's token (row t < 128) of the chunk at c0 of head h: its decay
// (1 past the head's end, or for threads t >= 128).  Loaded a chunk ahead of
// its use, so the load is not on the chunk's critical path.
__device__ __forceinline__ float row_decay(const FwdParams& p, int h, int c0, int valid) {
    const int t = threadIdx.x;
    if (t >= L || t >= valid) return 1.f;
    return p.gates ? __ldg(p.gates + static_cast<size_t>(h) * p.N + c0 + t)
                   : (p.gamma_head ? __ldg(p.gamma_head + h % p.H) : 1.f);
}

// dec[i] = sum of log2(decay) over the chunk's tokens 0 .. i, from each row's
// decay `gam` (row_decay).  Threads 0 .. 127 scan; every thread of the CTA
// calls it, and it ends with the scan complete for all of them.
__device__ __forceinline__ void decay_scan(float* dec, float gam) {
    const int t = threadIdx.x;
    float* wsum = dec + L;
    float l = 0.f;
    if (t < L) {
        l = log2_decay(gam);
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const float x = __shfl_up_sync(0xffffffffu, l, o);
            if ((t & 31) >= o) l += x;
        }
        if ((t & 31) == 31) wsum[t >> 5] = l;
    }
    __syncthreads();
    if (t < L) {
        for (int w = 0; w < (t >> 5); ++w) l += wsum[w];
        dec[t] = l;
    }
    __syncthreads();
}

// Row `row` of atom `a` of a K-major 128-row bf16 tile, times f (rounded to
// bf16), written to the same place in `dst` (which may be `tile`).
__device__ __forceinline__ void scale_row_atom_to(const uint8_t* tile, uint8_t* dst, int a, int row, float f) {
#pragma unroll
    for (int c = 0; c < 8; ++c) {
        const uint4 u = *reinterpret_cast<const uint4*>(tile + a * kAtom + swz(row, c));
        uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int k = 0; k < 4; ++k)
            w[k] = pack_bf16(__uint_as_float(w[k] << 16) * f, __uint_as_float(w[k] & 0xFFFF0000u) * f);
        *reinterpret_cast<uint4*>(dst + a * kAtom + swz(row, c)) = make_uint4(w[0], w[1], w[2], w[3]);
    }
}

// Row `row` of a K-major 128-row bf16 tile, atom `a`, times f (rounded to bf16).
__device__ __forceinline__ void scale_row_atom(uint8_t* tile, int a, int row, float f) {
#pragma unroll
    for (int c = 0; c < 8; ++c) {
        uint4* q = reinterpret_cast<uint4*>(tile + a * kAtom + swz(row, c));
        uint4 u = *q;
        uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int k = 0; k < 4; ++k)
            w[k] = pack_bf16(__uint_as_float(w[k] << 16) * f, __uint_as_float(w[k] & 0xFFFF0000u) * f);
        *q = make_uint4(w[0], w[1], w[2], w[3]);
    }
}

template <int D, int M, bool RET>
__global__ void __launch_bounds__(Layout<D, M, RET>::THREADS, Layout<D, M, RET>::PER_SM)
causal_fwd_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                     const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO,
                     const FwdParams p) {
    using Lay = Layout<D, M, RET>;
    constexpr int DA = Lay::DA, MA = Lay::MA, NE = Lay::NE, W = Lay::W, NT = Lay::THREADS;
    // retention at D = 64: the output staging tile takes one of the P area's two atoms, so the
    // other holds a decayed copy of K and the state update need not wait for the P epilogue
    constexpr bool KCOPY = RET && D == 64 && MA == 1;
    constexpr int HALF = M / Lay::GROUPS;   // columns of a state/output row per warpgroup
    constexpr int PCOLS = L / Lay::GROUPS;  // columns of P per warpgroup
    constexpr uint32_t ID_P = idesc_bf16(128, 128, false, false);
    constexpr uint32_t ID_S = idesc_bf16(128, NE, true, true);
    constexpr uint32_t ID_SV = idesc_bf16(128, M, true, true);   // phi(K)^T V
    constexpr uint32_t ID_S1 = idesc_bf16(128, 16, true, true);  // phi(K)^T 1
    constexpr uint32_t ID_O = idesc_bf16(128, NE, false, true);

    extern __shared__ __align__(1024) uint8_t sm[];
    float* const dec = reinterpret_cast<float*>(sm + Lay::DEC);  // retention: the chunk's a_i
    const int t = threadIdx.x, warp = t >> 5;
    const int q = warp & 3, g = warp >> 2;  // TMEM lane quarter, warpgroup
    const int row = 32 * q + (t & 31);      // tile row / TMEM lane owned by this thread
    if (smem_u32(sm) & 1023u) {  // the swizzled layouts need a 1024-aligned base
        if (t == 0) atomicOr(p.status, kErrAlign);
        return;
    }
    uint64_t* tma_bar = reinterpret_cast<uint64_t*>(sm + Lay::BARS);
    uint64_t* mma_bar = tma_bar + 1;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tma_bar + 2);
    volatile int* sh = reinterpret_cast<volatile int*>(tma_bar + 3);  // [0] unit, [1] abort
    uint64_t* kv_bar1 = tma_bar + 4;  // phase 1's copies into its second and third K, V buffers
    uint64_t* kv_bar2 = tma_bar + 5;
    volatile int* lb = reinterpret_cast<volatile int*>(tma_bar + 6);  // the look-back's result

    if (t == 0) {
        mbar_init(tma_bar, 1);
        mbar_init(mma_bar, 1);
        mbar_init(kv_bar1, 1);
        mbar_init(kv_bar2, 1);
        fence_mbar_init();
        sh[1] = 0;
    }
    if (warp == 0) {
        tmem_alloc(tmem_slot, Lay::T_COLS);
        tmem_relinquish();
    }
    for (int i = t; i < static_cast<int>(kAtom / 16); i += NT)  // bf16 1.0 everywhere
        reinterpret_cast<uint4*>(sm + Lay::ONES)[i] =
            make_uint4(0x3F803F80u, 0x3F803F80u, 0x3F803F80u, 0x3F803F80u);
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tm = *tmem_slot;
    if (t == 0) sh[0] = static_cast<int>(atomicAdd(p.ticket, 1u));
    __syncthreads();

    const int unit = sh[0];
    const UnitRange ur(unit, p.per, p.CH, p.BH);
    const uint32_t lane = static_cast<uint32_t>(32 * q) << 16;
    const uint32_t sQ = smem_u32(sm + Lay::Q), sK = smem_u32(sm + Lay::K);
    const uint32_t sV = smem_u32(sm + Lay::V);
    const uint32_t sS = smem_u32(sm + Lay::S);
    uint32_t mma_phase = 0;
    // thread 0's copies issued on, and waits completed on, each copy barrier (tma_bar doubles
    // as phase 1's first K, V buffer's), so that a CTA ending early drains what is in flight
    uint32_t put0 = 0, put1 = 0, put2 = 0, got0 = 0, got1 = 0, got2 = 0;
    float gam_next = 1.f;  // retention: this thread's row decay of the next chunk, loaded ahead
    bool fact = false;     // retention: the chunk's decays factor into its Q and K rows

    auto fail = [&](unsigned code) {
        atomicOr(p.status, code);
        sh[1] = 1;
    };
    // One thread polls the barrier; the others wait at the CTA barrier.
    auto wait_bar = [&](uint64_t* bar, uint32_t& phase) {
        if (t == 0 && !mbar_wait(bar, phase, kWaitLimit)) fail(kErrWait);
        __syncthreads();
        phase ^= 1u;
    };
    auto load = [&](int h, int c0, bool with_q) {  // thread 0 only
        ++put0;
        mbar_arrive_expect_tx(tma_bar, with_q ? Lay::TX_QKV : Lay::TX_KV);
        for (int a = 0; a < DA; ++a) {
            if (with_q) tma_load_3d(sm + Lay::Q + a * kAtom, &tmQ, tma_bar, 64 * a, c0, h);
            tma_load_3d(sm + Lay::K + a * kAtom, &tmK, tma_bar, 64 * a, c0, h);
        }
        for (int a = 0; a < MA; ++a)
            tma_load_3d(sm + Lay::V + a * kAtom, &tmV, tma_bar, 64 * a, c0, h);
    };
    // S_ext (+)= phi(K)^T [V | 1] from K at sk and V at sv (the ones atom kAtom * MA after it)
    auto mma_state_update = [&](uint32_t sk, uint32_t sv, bool accumulate_first) {
#pragma unroll
        for (int k = 0; k < L / 16; ++k)
            mma_bf16(tm + Lay::T_S, sdesc(sk + 2048 * k, kAtom, 1024),
                     sdesc(sv + 2048 * k, kAtom, 1024), ID_S, (accumulate_first || k > 0) ? 1u : 0u);
    };
    // Starting state of a segment of head h: the published aggregates of units
    // sp0 <= sp < sp1, on top of the inclusive state of unit sp0 - 1 when
    // `from_incl` (else the carried-in state), into TMEM and the bf16 S tile
    // (threads with q < D / 32: state row d = row).  With RET each term is decayed
    // by the pieces after it.
    auto put_state = [&](int h, int sp0, int sp1, bool from_incl) {
        const float* base = from_incl ? p.incl + static_cast<size_t>(sp0 - 1) * W : nullptr;
        const int d = row;
        for (int j0 = g * HALF; j0 < (g + 1) * HALF; j0 += 16) {
            float v[16];
            if constexpr (RET) {  // each aggregate decayed by the pieces after it, then S_init
                float f = 1.f;
#pragma unroll
                for (int i = 0; i < 16; ++i) v[i] = 0.f;
                for (int sp = sp1 - 1; sp >= sp0; --sp) {
                    const float4* a =
                        reinterpret_cast<const float4*>(p.agg + static_cast<size_t>(sp) * W + d * M + j0);
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const float4 x = __ldcg(a + u);
                        v[4 * u] = fmaf(f, x.x, v[4 * u]);
                        v[4 * u + 1] = fmaf(f, x.y, v[4 * u + 1]);
                        v[4 * u + 2] = fmaf(f, x.z, v[4 * u + 2]);
                        v[4 * u + 3] = fmaf(f, x.w, v[4 * u + 3]);
                    }
                    f *= exp2f(__ldcg(p.lam + sp));
                }
                if (base)
#pragma unroll
                    for (int i = 0; i < 16; ++i) v[i] = fmaf(f, __ldcg(base + d * M + j0 + i), v[i]);
                else if (p.S_init)
#pragma unroll
                    for (int i = 0; i < 16; ++i)
                        v[i] = fmaf(f, p.S_init[(static_cast<size_t>(h) * D + d) * M + j0 + i], v[i]);
            } else {
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    v[i] = base ? __ldcg(base + d * M + j0 + i)
                                : (p.S_init ? p.S_init[(static_cast<size_t>(h) * D + d) * M + j0 + i] : 0.f);
                for (int sp = sp0; sp < sp1; ++sp) {
                    const float4* a =
                        reinterpret_cast<const float4*>(p.agg + static_cast<size_t>(sp) * W + d * M + j0);
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const float4 x = __ldcg(a + u);
                        v[4 * u] += x.x;
                        v[4 * u + 1] += x.y;
                        v[4 * u + 2] += x.z;
                        v[4 * u + 3] += x.w;
                    }
                }
            }
            tmem_st16(tm + lane + Lay::T_S + j0, v);
            const int cc = j0 >> 3;
            *reinterpret_cast<uint4*>(sm + Lay::S + (cc >> 3) * Lay::S_ATOM + swz(d, cc & 7)) =
                make_uint4(pack_bf16(v[0], v[1]), pack_bf16(v[2], v[3]), pack_bf16(v[4], v[5]),
                           pack_bf16(v[6], v[7]));
            *reinterpret_cast<uint4*>(sm + Lay::S + ((cc + 1) >> 3) * Lay::S_ATOM +
                                      swz(d, (cc + 1) & 7)) =
                make_uint4(pack_bf16(v[8], v[9]), pack_bf16(v[10], v[11]), pack_bf16(v[12], v[13]),
                           pack_bf16(v[14], v[15]));
        }
        if (g == 0) {  // Z (read only without RET, where it is the normaliser state)
            float z = base ? __ldcg(base + D * M + d) : (p.Z_init ? p.Z_init[static_cast<size_t>(h) * D + d] : 0.f);
            for (int sp = sp0; sp < sp1; ++sp) z += __ldcg(p.agg + static_cast<size_t>(sp) * W + D * M + d);
            float zv[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) zv[i] = z;
            tmem_st16(tm + lane + Lay::T_S + M, zv);
            const uint32_t zz = pack_bf16(z, z);
            const uint4 z4 = make_uint4(zz, zz, zz, zz);
            *reinterpret_cast<uint4*>(sm + Lay::S + MA * Lay::S_ATOM + swz(d, 0)) = z4;
            *reinterpret_cast<uint4*>(sm + Lay::S + MA * Lay::S_ATOM + swz(d, 1)) = z4;
        }
    };

    // ------------------------- phase 1: aggregate of a last segment that stops mid-head
    // K and V go round three buffers: their own tiles, the idle Q and P areas, and the
    // third buffer of the layout (the S area is idle too), so two copies are in flight while a
    // chunk is summed.  V no longer sits before the ones atom there, so the normaliser column takes
    // its own N = 16 product against the ones atom.
    if (ur.publish) {
        constexpr int KV_BUFS = 3;
        const int h = ur.hB, g0 = max(ur.start, h * p.CH);
        auto k_buf = [](int b) { return b == 0 ? Lay::K : b == 1 ? Lay::Q : Lay::KV2_K; };
        auto v_buf = [](int b) { return b == 0 ? Lay::V : b == 1 ? Lay::P : Lay::KV2_V; };
        auto kv_bar = [&](int b) { return b == 0 ? tma_bar : b == 1 ? kv_bar1 : kv_bar2; };
        auto load_kv = [&](int c0, int b) {  // thread 0 only
            put0 += b == 0;
            put1 += b == 1;
            put2 += b == 2;
            mbar_arrive_expect_tx(kv_bar(b), Lay::TX_KV);
            for (int a = 0; a < DA; ++a)
                tma_load_3d(sm + k_buf(b) + a * kAtom, &tmK, kv_bar(b), 64 * a, c0, h);
            for (int a = 0; a < MA; ++a)
                tma_load_3d(sm + v_buf(b) + a * kAtom, &tmV, kv_bar(b), 64 * a, c0, h);
        };
        const uint32_t sOnes = smem_u32(sm + Lay::ONES);
        // The chunks are summed last to first: the ones phase 2 reads first are then the most
        // recently read, and still in L2.
        const int n1 = ur.end - g0;
        const int c_last = (ur.end - 1 - h * p.CH) * L;  // the first chunk summed
        if (t == 0)
            for (int b = 0; b < KV_BUFS - 1 && b < n1; ++b) load_kv(c_last - b * L, b);
        float run = 0.f;  // retention: log2 decay of the piece's chunks already summed (the later ones)
        if (RET) gam_next = row_decay(p, h, c_last, min(L, p.N - c_last));
        for (int i1 = 0; i1 < n1; ++i1) {
            const int c0 = c_last - i1 * L;
            const int b = i1 % KV_BUFS;
            if (t == 0) {
                const uint32_t done = b == 0 ? got0 : b == 1 ? got1 : got2;
                if (!mbar_wait(kv_bar(b), done & 1u, kWaitLimit)) fail(kErrWait);
                got0 += b == 0;
                got1 += b == 1;
                got2 += b == 2;
            }
            __syncthreads();
            if (i1 > 0) {  // the previous chunk's MMA has released its buffer
                wait_bar(mma_bar, mma_phase);
                fence_after_sync();
            }
            if (t == 0 && i1 + KV_BUFS - 1 < n1)
                load_kv(c0 - (KV_BUFS - 1) * L, (i1 + KV_BUFS - 1) % KV_BUFS);
            if constexpr (RET) {  // K rows decayed to the end of the piece
                const float gam = gam_next;
                if (i1 + 1 < n1) gam_next = row_decay(p, h, c0 - L, L);
                decay_scan(dec, gam);
                const float A = dec[L - 1];
                const float f = exp2f(run + A - dec[row]);
                for (int a = g; a < DA; a += Lay::GROUPS) scale_row_atom(sm + k_buf(b), a, row, f);
                run += A;
            } else {
                phi_tile<true, NT>(sm + k_buf(b), DA, min(L, p.N - c0));
            }
            fence_proxy_async();
            fence_before_sync();
            __syncthreads();
            fence_after_sync();
            if (sh[1]) goto cleanup;
            if (t == 0) {
                const uint32_t sk = smem_u32(sm + k_buf(b)), sv = smem_u32(sm + v_buf(b));
#pragma unroll
                for (int k = 0; k < L / 16; ++k) {
                    const uint32_t acc = (i1 > 0 || k > 0) ? 1u : 0u;
                    const uint64_t a = sdesc(sk + 2048 * k, kAtom, 1024);
                    mma_bf16(tm + Lay::T_S, a, sdesc(sv + 2048 * k, kAtom, 1024), ID_SV, acc);
                    mma_bf16(tm + Lay::T_S + M, a, sdesc(sOnes + 2048 * k, kAtom, 1024), ID_S1, acc);
                }
                mma_commit(mma_bar);
            }
        }
        wait_bar(mma_bar, mma_phase);
        fence_after_sync();
        // a piece that starts at its head's start knows the head's state at its end now:
        // the carried-in state (decayed by the piece) plus the aggregate
        const bool incl_now = p.use_incl && g0 == h * p.CH;
        const float f_in = RET ? exp2f(run) : 1.f;
        if (q < D / 32) {  // rows d < D of S_ext, this warpgroup's columns
            float* out = p.agg + static_cast<size_t>(unit) * W;
            float* inc = p.incl + static_cast<size_t>(unit) * W;
            const int d = row;
            for (int j0 = g * HALF; j0 < (g + 1) * HALF; j0 += 32) {
                float v[32];
                tmem_ld32(tm + lane + Lay::T_S + j0, v);
#pragma unroll
                for (int u = 0; u < 8; ++u)
                    reinterpret_cast<float4*>(out + d * M + j0)[u] =
                        make_float4(v[4 * u], v[4 * u + 1], v[4 * u + 2], v[4 * u + 3]);
                if (incl_now) {
                    if (p.S_init) {
                        const float* si = p.S_init + (static_cast<size_t>(h) * D + d) * M + j0;
#pragma unroll
                        for (int u = 0; u < 32; ++u) v[u] = fmaf(f_in, si[u], v[u]);
                    }
#pragma unroll
                    for (int u = 0; u < 8; ++u)
                        reinterpret_cast<float4*>(inc + d * M + j0)[u] =
                            make_float4(v[4 * u], v[4 * u + 1], v[4 * u + 2], v[4 * u + 3]);
                }
            }
            if (g == 0) {
                float z[16];
                tmem_ld16(tm + lane + Lay::T_S + M, z);
                out[D * M + d] = z[0];
                if (incl_now) inc[D * M + d] = z[0] + (p.Z_init ? f_in * p.Z_init[static_cast<size_t>(h) * D + d] : 0.f);
            }
        }
        if (RET && t == 0) p.lam[unit] = run;
        __threadfence();
        fence_before_sync();
        __syncthreads();
        if (t == 0 && unit != p.withhold) st_release(p.flags + unit, incl_now ? 2u : 1u);
    }

    // phase 2's first copy goes out now, under the look-back (it touches no state tile or TMEM)
    if (t == 0) load(ur.hA, (ur.start - ur.hA * p.CH) * L, true);

    // ------------------ look-back: starting state of the first segment
    // Walks back from the unit before this one, waiting for each one's aggregate (flag 1),
    // and stops at the first whose inclusive state is there already (flag 2), or at the
    // head's first unit; no unit waits for an inclusive state, so a late one is never worse
    // off than summing every earlier aggregate.
    if (t == 0) {
        int sp0 = unit;  // the aggregates of units sp0 .. unit - 1 are summed
        int from_incl = 0;
        if (ur.look) {
            for (int sp = unit - 1; sp >= ur.u_first && !sh[1]; --sp) {
                uint32_t n = 0;
                unsigned fl;
                while ((fl = ld_acquire(p.flags + sp)) == 0u) {
                    if (++n > p.spin_limit) {
                        fail(kErrLookback);
                        break;
                    }
                    __nanosleep(256);
                }
                if (fl == 2u) {
                    sp0 = sp + 1;
                    from_incl = 1;
                    break;
                }
                sp0 = sp;
            }
        }
        lb[0] = sp0;
        lb[1] = from_incl;
    }
    __syncthreads();
    if (sh[1]) goto cleanup;
    if (q < D / 32) put_state(ur.hA, lb[0], unit, lb[1] != 0);
    fence_proxy_async();
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    // A unit that looked back and publishes a piece of the same head now knows the head's
    // state at its end: its starting state (decayed by its piece) plus its aggregate.
    if (p.use_incl && ur.look && ur.publish && ur.hA == ur.hB) {
        if (q < D / 32) {
            const float* a = p.agg + static_cast<size_t>(unit) * W;
            float* inc = p.incl + static_cast<size_t>(unit) * W;
            const float f = RET ? exp2f(__ldcg(p.lam + unit)) : 1.f;
            const int d = row;
            for (int j0 = g * HALF; j0 < (g + 1) * HALF; j0 += 32) {
                float v[32];
                tmem_ld32(tm + lane + Lay::T_S + j0, v);
#pragma unroll
                for (int u = 0; u < 32; ++u) v[u] = fmaf(f, v[u], __ldcg(a + d * M + j0 + u));
#pragma unroll
                for (int u = 0; u < 8; ++u)
                    reinterpret_cast<float4*>(inc + d * M + j0)[u] =
                        make_float4(v[4 * u], v[4 * u + 1], v[4 * u + 2], v[4 * u + 3]);
            }
            if (g == 0) {
                float z[16];
                tmem_ld16(tm + lane + Lay::T_S + M, z);
                inc[D * M + d] = fmaf(f, z[0], __ldcg(a + D * M + d));
            }
        }
        __threadfence();
        fence_before_sync();
        __syncthreads();
        if (t == 0 && unit != p.withhold) st_release(p.flags + unit, 2u);
    }

    // ------------------------------------------------- phase 2: outputs
    if (RET) {  // the first chunk's row decay
        const int h0 = ur.start / p.CH, c00 = (ur.start - h0 * p.CH) * L;
        gam_next = row_decay(p, h0, c00, min(L, p.N - c00));
    }
    for (int gc = ur.start; gc < ur.end; ++gc) {
        const int h = gc / p.CH, cc = gc - h * p.CH;
        const int c0 = cc * L;
        const int valid = min(L, p.N - c0);
        if (t == 0 && !mbar_wait(tma_bar, (got0++) & 1u, kWaitLimit)) fail(kErrWait);
        __syncthreads();
        if constexpr (RET) {
            const float gam = gam_next;
            if (gc + 1 < ur.end) {
                const int hn = (gc + 1) / p.CH, cn0 = (gc + 1 - hn * p.CH) * L;
                gam_next = row_decay(p, hn, cn0, min(L, p.N - cn0));
            }
            decay_scan(dec, gam);
            fact = dec[L - 1] >= kFactorMin;
            if (fact) {  // Q rows by 2^(a_i), K rows by 2^(-a_i): P comes out decayed
                const float ai = dec[row];
                for (int a = g; a < DA; a += Lay::GROUPS) {
                    scale_row_atom(sm + Lay::Q, a, row, exp2f(ai));
                    scale_row_atom(sm + Lay::K, a, row, exp2f(-ai));
                }
            } else if constexpr (KCOPY) {  // the decayed K rows into the spare staging atom and the
                                           // state times 2^A now, so the update can follow P at once
                const float A = dec[L - 1];
                scale_row_atom_to(sm + Lay::K, sm + Lay::P + kAtom, 0, row, exp2f(A - dec[row]));
                if (q < D / 32) {
                    const float f = exp2f(A);
                    for (int col = 0; col < NE; col += 16) {
                        float v[16];
                        tmem_ld16(tm + lane + Lay::T_S + col, v);
#pragma unroll
                        for (int i = 0; i < 16; ++i) v[i] *= f;
                        tmem_st16(tm + lane + Lay::T_S + col, v);
                    }
                }
            }
        } else {
            phi_tile<false, NT>(sm + Lay::Q, DA, valid);
            phi_tile<true, NT>(sm + Lay::K, DA, valid);
        }
        fence_proxy_async();
        fence_before_sync();
        __syncthreads();
        fence_after_sync();
        if (sh[1]) goto cleanup;
        if (t == 0) {
#pragma unroll
            for (int k = 0; k < D / 16; ++k) {
                const uint32_t off = (k >> 2) * kAtom + 32 * (k & 3);
                mma_bf16(tm + Lay::T_P, sdesc(sQ + off, 16, 1024), sdesc(sK + off, 16, 1024), ID_P,
                         k > 0 ? 1u : 0u);
            }
            mma_commit(mma_bar);
            if (!RET || fact) mma_state_update(sK, sV, true);  // under the P epilogue; tracked by the next commit
            else if (KCOPY) mma_state_update(smem_u32(sm + Lay::P + kAtom), sV, true);  // decayed K copy
            tma_store_wait_read();           // the staging tile (P area) is free again
        }
        wait_bar(mma_bar, mma_phase);
        fence_after_sync();
        {   // P: mask j > i, round to bf16 pairs, pack in place in TMEM (each 64 columns read
            // before their 32 packed ones are written over the first half of them)
#pragma unroll
            for (int jb = 0; jb < PCOLS / 64; ++jb) {
                const int j0 = g * PCOLS + jb * 64;
                uint32_t pk[32];
                if (j0 > 32 * q + 31) {
#pragma unroll
                    for (int u = 0; u < 32; ++u) pk[u] = 0u;
                } else {
                    float v[64];
                    tmem_ld64(tm + lane + Lay::T_P + j0, v);
                    if (RET && !fact) {  // decay 2^(a_i - a_j) of key j seen from query i
                        const float ai = dec[row];
#pragma unroll
                        for (int u = 0; u < 32; ++u) {
                            const int j = j0 + 2 * u;
                            pk[u] = pack_bf16(j <= row ? v[2 * u] * exp2f(ai - dec[j]) : 0.f,
                                              j + 1 <= row ? v[2 * u + 1] * exp2f(ai - dec[j + 1]) : 0.f);
                        }
                    } else {
#pragma unroll
                        for (int u = 0; u < 32; ++u) {
                            const int j = j0 + 2 * u;
                            pk[u] = pack_bf16(j <= row ? v[2 * u] : 0.f, j + 1 <= row ? v[2 * u + 1] : 0.f);
                        }
                    }
                }
                tmem_st32u(tm + lane + Lay::T_P + g * PCOLS + 32 * jb, pk);
            }
        }
        if (RET && !fact) {  // P is taken: Q rows by 2^(a_i), K rows by 2^(A - a_j), the state by 2^A
            const float A = dec[L - 1], ai = dec[row];
            for (int a = g; a < DA; a += Lay::GROUPS) {
                scale_row_atom(sm + Lay::Q, a, row, exp2f(ai));
                if (!KCOPY) scale_row_atom(sm + Lay::K, a, row, exp2f(A - ai));
            }
            if (!KCOPY && q < D / 32) {
                const float f = exp2f(A);
                for (int j0 = g * HALF; j0 < (g + 1) * HALF + (g == 0 ? 16 : 0); j0 += 16) {
                    const int col = j0 < (g + 1) * HALF ? j0 : M;  // then the normaliser block
                    float v[16];
                    tmem_ld16(tm + lane + Lay::T_S + col, v);
#pragma unroll
                    for (int i = 0; i < 16; ++i) v[i] *= f;
                    tmem_st16(tm + lane + Lay::T_S + col, v);
                }
            }
            fence_proxy_async();  // the rescaled Q and K rows, for the products below
        }
        fence_before_sync();
        __syncthreads();
        fence_after_sync();
        if (t == 0) {
            if (RET && !KCOPY && !fact) mma_state_update(sK, sV, true);  // with the decayed K rows
#pragma unroll
            for (int k = 0; k < D / 16; ++k)  // O_ext = phi(Q) [S | Z]
                mma_bf16(tm + Lay::T_O, sdesc(sQ + (k >> 2) * kAtom + 32 * (k & 3), 16, 1024),
                         sdesc(sS + 2048 * k, Lay::S_ATOM, 1024), ID_O, k > 0 ? 1u : 0u);
#pragma unroll
            for (int k = 0; k < L / 16; ++k)  // O_ext += P [V | 1], P read from TMEM
                mma_bf16_ts(tm + Lay::T_O, tm + Lay::T_P + Lay::p_col(k), sdesc(sV + 2048 * k, kAtom, 1024),
                            ID_O, 1u);
            mma_commit(mma_bar);
        }
        wait_bar(mma_bar, mma_phase);
        fence_after_sync();
        if (t == 0 && gc + 1 < ur.end) {  // every input tile is consumed
            const int hn = (gc + 1) / p.CH;
            load(hn, (gc + 1 - hn * p.CH) * L, true);
        }
        if (q < D / 32) {
            const int d = row;
            // factored decays: the state in TMEM is S_{c-1} + (K rows by 2^(-a))^T [V | 1], the
            // chunk's state 2^A times that; scaled as it is read, and written back for the next chunk
            const float fA = RET && fact ? exp2f(dec[L - 1]) : 1.f;
            auto state32 = [&](int j0, float (&v)[32], bool write_back) {
                tmem_ld32(tm + lane + Lay::T_S + j0, v);
                if (RET && fact) {
#pragma unroll
                    for (int u = 0; u < 32; ++u) v[u] *= fA;
                    if (write_back) tmem_st32u(tm + lane + Lay::T_S + j0, reinterpret_cast<const uint32_t(&)[32]>(v));
                }
            };
            auto state_z = [&](float (&z)[16], bool write_back) {
                tmem_ld16(tm + lane + Lay::T_S + M, z);
                if (RET && fact) {
#pragma unroll
                    for (int u = 0; u < 16; ++u) z[u] *= fA;
                    if (write_back) tmem_st16(tm + lane + Lay::T_S + M, z);
                }
            };
            if (cc == p.CH - 1) {  // the head ends here: its final state, then the next head's start
                if (p.S_final) {
                    float* so = p.S_final + (static_cast<size_t>(h) * D + d) * M;
                    for (int j0 = g * HALF; j0 < (g + 1) * HALF; j0 += 32) {
                        float v[32];
                        state32(j0, v, false);
#pragma unroll
                        for (int u = 0; u < 8; ++u)
                            reinterpret_cast<float4*>(so + j0)[u] =
                                make_float4(v[4 * u], v[4 * u + 1], v[4 * u + 2], v[4 * u + 3]);
                    }
                    if (g == 0 && p.Z_final) {
                        float z[16];
                        state_z(z, false);
                        p.Z_final[static_cast<size_t>(h) * D + d] = z[0];
                    }
                }
                if (gc + 1 < ur.end) put_state(h + 1, 0, 0, false);
            } else {  // S_c -> bf16 copy for the next chunk's O_ext (and a checkpoint)
                float* ck = p.ckpt && (cc + 1) % kCkptChunks == 0
                                ? p.ckpt + (static_cast<size_t>(h) * ckpt_slots(p.CH) + (cc + 1) / kCkptChunks) * W
                                : nullptr;
                for (int j0 = g * HALF; j0 < (g + 1) * HALF; j0 += 32) {
                    float v[32];
                    state32(j0, v, true);
                    if (ck) {
#pragma unroll
                        for (int u = 0; u < 8; ++u)
                            reinterpret_cast<float4*>(ck + d * M + j0)[u] =
                                make_float4(v[4 * u], v[4 * u + 1], v[4 * u + 2], v[4 * u + 3]);
                    }
                    uint32_t pk[16];
#pragma unroll
                    for (int u = 0; u < 16; ++u) pk[u] = pack_bf16(v[2 * u], v[2 * u + 1]);
                    store_row32(sm + Lay::S, Lay::S_ATOM, d, j0, pk);
                }
                if (g == 0) {
                    float z[16];
                    state_z(z, true);
                    if (ck) ck[D * M + d] = z[0];
                    uint32_t zk[8];
#pragma unroll
                    for (int u = 0; u < 8; ++u) zk[u] = pack_bf16(z[2 * u], z[2 * u + 1]);
                    *reinterpret_cast<uint4*>(sm + Lay::S + MA * Lay::S_ATOM + swz(d, 0)) =
                        make_uint4(zk[0], zk[1], zk[2], zk[3]);
                    *reinterpret_cast<uint4*>(sm + Lay::S + MA * Lay::S_ATOM + swz(d, 1)) =
                        make_uint4(zk[4], zk[5], zk[6], zk[7]);
                }
            }
        }
        {   // V' = O_ext[:, :M] / O_ext[:, M] -> bf16 staging tile (P area)
            float dv[16];
            tmem_ld16(tm + lane + Lay::T_O + M, dv);
            const float inv = RET ? 1.f : 1.f / dv[0];  // retention has no normaliser
            if (p.den && g == 0 && row < valid) p.den[static_cast<size_t>(h) * p.N + c0 + row] = dv[0];
            for (int j0 = g * HALF; j0 < (g + 1) * HALF; j0 += 32) {
                float v[32];
                tmem_ld32(tm + lane + Lay::T_O + j0, v);
                uint32_t pk[16];
#pragma unroll
                for (int u = 0; u < 16; ++u) pk[u] = pack_bf16(v[2 * u] * inv, v[2 * u + 1] * inv);
                store_row32(sm + Lay::P, kAtom, row, j0, pk);
            }
        }
        fence_proxy_async();
        fence_before_sync();
        __syncthreads();
        fence_after_sync();
        if (t == 0) {
            for (int a = 0; a < MA; ++a) tma_store_3d(&tmO, sm + Lay::P + a * kAtom, 64 * a, c0, h);
            tma_store_commit();
        }
    }

cleanup:
    if (t == 0) {  // copies still in flight after an early exit land before the CTA leaves
        for (; got0 < put0; ++got0) mbar_wait(tma_bar, got0 & 1u, kWaitLimit);
        for (; got1 < put1; ++got1) mbar_wait(kv_bar1, got1 & 1u, kWaitLimit);
        for (; got2 < put2; ++got2) mbar_wait(kv_bar2, got2 & 1u, kWaitLimit);
        tma_store_wait_all();
    }
    fence_before_sync();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tm, Lay::T_COLS);
}

}  // namespace tcf

size_t causal_forward_tc_scratch(int D, int BH, int N, int num_sms) {
    using namespace tcf;
    const int per_sm = D == 64 ? Layout<64, 64>::PER_SM : Layout<128, 128>::PER_SM;
    const int chunks = (N + L - 1) / L;
    const size_t units = static_cast<size_t>(plan::tc_units(BH, chunks, per_sm * num_sms));
    // aggregates and inclusive states, flags and the ticket
    return 2 * sizeof(float) * units * plan::state_words(D, D) + sizeof(unsigned) * (units + 1) + 256;
}

size_t retention_forward_tc_scratch(int D, int BH, int N, int num_sms) {
    using namespace tcf;
    const int per_sm = D == 64 ? Layout<64, 64, true>::PER_SM : Layout<128, 128, true>::PER_SM;
    const int chunks = (N + L - 1) / L;
    const size_t units = static_cast<size_t>(plan::tc_units(BH, chunks, per_sm * num_sms));
    // the causal forward's aggregates, inclusive states and flags, plus one total log2 decay per unit
    return sizeof(float) * units * (2 * plan::state_words(D, D) + 1) + sizeof(unsigned) * (units + 1) + 256;
}

namespace tcf {

// Launches the forward kernel (RET: retention) with the split and scratch of `p`'s sizes.
template <int D, int M, bool RET>
cudaError_t launch_forward(const LaunchCtx& c, const __nv_bfloat16* Q, const __nv_bfloat16* K,
                           const __nv_bfloat16* V, __nv_bfloat16* O, int BH, int N, FwdParams p) {
    using Lay = Layout<D, M, RET>;
    const int chunks = (N + L - 1) / L;
    auto kern = causal_fwd_tc_kernel<D, M, RET>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(Lay::BYTES));
    if (e == cudaSuccess)  // all of the unified L1/shared storage as shared memory
        e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                                 cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, Lay::THREADS, Lay::BYTES);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) return cudaErrorInvalidConfiguration;
    // The occupancy query does not see the carve-out the driver picks at launch
    // and can report one CTA where two fit, so the split uses the fit computed
    // from shared memory and TMEM.  (Correctness does not depend on it: a CTA
    // only ever waits for CTAs that took their ticket, and so started, before it.)
    const int slots = Lay::PER_SM * c.num_sms;  // CTAs resident at once
    const ChunkSplit split = split_chunks(BH, chunks, slots);
    const int units = split.units;

    const size_t agg_bytes = sizeof(float) * static_cast<size_t>(units) * Lay::W;
    const size_t flag_bytes = sizeof(unsigned) * (static_cast<size_t>(units) + 1);
    const size_t bytes = RET ? retention_forward_tc_scratch(D, BH, N, c.num_sms)
                             : causal_forward_tc_scratch(D, BH, N, c.num_sms);
    char* ws = nullptr;
    e = scratch_alloc(c, reinterpret_cast<void**>(&ws), bytes);
    if (e != cudaSuccess) return e;
    p.N = N;
    p.BH = BH;
    p.CH = chunks;
    p.per = split.per;
    p.agg = reinterpret_cast<float*>(ws);
    p.incl = reinterpret_cast<float*>(ws + agg_bytes);
    // Measured: with many ranges per head a late range's walk over every earlier aggregate
    // dominates (one 262144-token head at D = 64, 292 ranges: 0.50 -> 0.38 ms with the end
    // states); with 64 ranges per head the extra publication costs 3% more than it saves, and
    // at D = 128 (66 KB end states) 4-6%.
    p.use_incl = D == 64 && chunks / split.per > 128;
    p.flags = reinterpret_cast<unsigned*>(ws + 2 * agg_bytes);
    p.ticket = p.flags + units;
    p.lam = RET ? reinterpret_cast<float*>(ws + 2 * agg_bytes + flag_bytes) : nullptr;
    p.withhold = c.withhold_unit;
    p.spin_limit = c.spin_limit ? c.spin_limit : kSpinLimit;
    p.status = c.status_word;
    do {
        if ((e = cudaMemsetAsync(p.flags, 0, flag_bytes, c.stream)) != cudaSuccess) break;
        CUtensorMap mQ, mK, mV, mO;
        if ((e = make_map(&mQ, Q, BH, N, D)) || (e = make_map(&mK, K, BH, N, D)) ||
            (e = make_map(&mV, V, BH, N, M)) || (e = make_map(&mO, O, BH, N, M)))
            break;
        kern<<<units, Lay::THREADS, Lay::BYTES, c.stream>>>(mQ, mK, mV, mO, p);
        note_launch();
        e = cudaGetLastError();
    } while (0);
    scratch_free(c, ws);
    return e;
}

}  // namespace tcf

template <int D, int M>
cudaError_t causal_forward_tc(const LaunchCtx& c, const __nv_bfloat16* Q, const __nv_bfloat16* K,
                              const __nv_bfloat16* V, __nv_bfloat16* O, int BH, int N,
                              const float* S_init, const float* Z_init, float* S_final,
                              float* Z_final, float* Den, float* Ckpt) {
    tcf::FwdParams p{};
    p.S_init = S_init;
    p.Z_init = Z_init;
    p.S_final = S_final;
    p.Z_final = Z_final;
    p.den = Den;
    p.ckpt = Ckpt;
    return tcf::launch_forward<D, M, false>(c, Q, K, V, O, BH, N, p);
}

template <int D, int M>
cudaError_t retention_forward_tc(const LaunchCtx& c, const __nv_bfloat16* Q, const __nv_bfloat16* K,
                                 const __nv_bfloat16* V, __nv_bfloat16* O, const float* gamma_head,
                                 const float* gates, int BH, int H, int N, const float* S_init,
                                 float* S_final) {
    tcf::FwdParams p{};
    p.S_init = S_init;
    p.S_final = S_final;
    p.gates = gates;
    p.gamma_head = gamma_head;
    p.H = H;
    return tcf::launch_forward<D, M, true>(c, Q, K, V, O, BH, N, p);
}

template cudaError_t retention_forward_tc<64, 64>(const LaunchCtx&, const __nv_bfloat16*,
                                                  const __nv_bfloat16*, const __nv_bfloat16*,
                                                  __nv_bfloat16*, const float*, const float*, int,
                                                  int, int, const float*, float*);
template cudaError_t retention_forward_tc<128, 128>(const LaunchCtx&, const __nv_bfloat16*,
                                                    const __nv_bfloat16*, const __nv_bfloat16*,
                                                    __nv_bfloat16*, const float*, const float*, int,
                                                    int, int, const float*, float*);
template cudaError_t causal_forward_tc<64, 64>(const LaunchCtx&, const __nv_bfloat16*,
                                               const __nv_bfloat16*, const __nv_bfloat16*,
                                               __nv_bfloat16*, int, int, const float*, const float*,
                                               float*, float*, float*, float*);
template cudaError_t causal_forward_tc<128, 128>(const LaunchCtx&, const __nv_bfloat16*,
                                                 const __nv_bfloat16*, const __nv_bfloat16*,
                                                 __nv_bfloat16*, int, int, const float*,
                                                 const float*, float*, float*, float*, float*);

}  // namespace la
