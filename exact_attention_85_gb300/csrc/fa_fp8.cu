// fa_fp8.cu -- FP8 (e4m3) path for sm_103a: random-sign Hadamard rotation
// with per-tensor quantisation, and the FP8 forward.
//
// From the FlashAttention-3 summary page (vi.news.hada.io), "FP8" and
// "incoherent processing": FP8 doubles tensor-core throughput; outliers in
// Q and K inflate the quantisation error, which is reduced by multiplying Q
// and K by a random orthogonal matrix -- a Hadamard transform with random
// signs, O(d log d) per row -- which leaves Q K^T unchanged.
//
// Quantisation (two passes over the tensor, both memory bound):
//   hq_amax_kernel   x' = (x o s) H_d / sqrt(d) per row (fast Walsh-Hadamard
//                    butterflies in registers and warp shuffles), amax |x'|
//   hq_quant_kernel  recomputes x', x8 = e4m3(x' * 448 / amax) (round to
//                    nearest even, saturating), descale = amax / 448
// With signs == NULL the rotation is skipped (plain per-tensor FP8).
//
// Forward (fwd_fp8_kernel): the structure of the bf16 forward (fa_fwd.cu,
// two Q tiles per CTA) with kind::f8f6f4 MMAs: Q, K, V e4m3 in 128-byte-swizzled shared memory
// (one 128-byte row = 128 values, so d = 128 is one swizzle atom wide), P
// quantised to e4m3 in tensor memory as the A operand of O += P V.  Scores are
// descaled as S = scale * q_descale * k_descale * Q8 K8^T; O is multiplied by
// v_descale in the epilogue.  P is lifted by 2^4 before quantisation so its
// typical values sit in e4m3's normal range; the running max moves when a
// tile's max exceeds it by more than 4 (log2 units), so P <= 2^8 < 448.  O is
// normalised by a sum of the quantised P it was built from, so the lift
// cancels; that sum is accumulated in fp16 pairs (8 values per half before it
// is widened), whose 11-bit significand rounds it by at most about 2^-11
// relative per add -- far below the 2^-4 rounding of P itself.  L uses the
// fp32 sum of the unquantised P.
#include "grid_order.cuh"
#include "host_util.h"
#include "ptx.cuh"

namespace fa {

namespace {

// ------------------------------------------------------------ e4m3 helpers

// Two floats -> two e4m3 bytes (round to nearest even, saturating); `lo` in
// bits 0-7.
__device__ __forceinline__ uint32_t cvt_e4m3x2(float lo, float hi) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

// Two e4m3 bytes (bits 0-15) -> two fp16 values (exact), packed.
__device__ __forceinline__ uint32_t e4m3x2_to_h2(uint32_t v) {
    uint32_t h2;
    const uint16_t in = (uint16_t)v;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(in));
    return h2;
}

// Two e4m3 bytes (bits 0-15) -> two floats (exact).
__device__ __forceinline__ float2 e4m3x2_to_float2(uint32_t v) {
    uint32_t h2;
    const uint16_t in = (uint16_t)v;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(in));
    float lo, hi;
    asm("{\n\t.reg .b16 a, b;\n\tmov.b32 {a, b}, %2;\n\t"
        "cvt.f32.f16 %0, a;\n\tcvt.f32.f16 %1, b;\n\t}\n"
        : "=f"(lo), "=f"(hi)
        : "r"(h2));
    return make_float2(lo, hi);
}

// --------------------------------------------- Hadamard + quantise kernels
// Row layout: 4 lanes per row; lane j (0..3) holds the 16-byte chunks
// 4 k + j (k = 0 .. D/32 - 1) of its row, 8 values each, so a warp holds 8
// rows and every load instruction covers 64 contiguous bytes of each row.
// In the row index v = 8 (4 k + j) + e the butterflies for the bits of e and
// of k run inside a lane, those for the two bits of j across the 4 lanes (2
// shuffle stages; with one chunk per lane and 16 lanes per row it took 4).

template <int D>
struct HqShape {
    static constexpr int CPL = D / 32;   // 16-byte chunks per lane
    static constexpr int VPL = CPL * 8;  // values per lane
    static constexpr int RPW = 8;        // rows per warp
    // groups of 8 rows per warp and trip, all loaded before any is
    // transformed, so several loads per warp are in flight
    static constexpr int KU = D == 128 ? 2 : 4;
};

// The transform on packed pairs w[p] = (v[2p], v[2p + 1]): stride 1 inside a
// pair, strides >= 2 as packed fp32 adds of whole pairs, the two cross-lane
// stages as one packed fma each (x + other, or other - x in the upper lane).
// On bf16 inputs every partial sum is exact in fp32, so any stage order
// gives the same result.  The 1/sqrt(d) factor is left to the caller.
template <int D>
__device__ __forceinline__ void hadamard_pairs(float2 (&w)[HqShape<D>::VPL / 2], int j) {
    constexpr int NP = HqShape<D>::VPL / 2;
#pragma unroll
    for (int p = 0; p < NP; ++p) {
        const float a = w[p].x, b = w[p].y;
        w[p] = make_float2(a + b, a - b);
    }
#pragma unroll
    for (int s = 1; s < NP; s <<= 1) {
#pragma unroll
        for (int p = 0; p < NP; ++p) {
            if ((p & s) == 0) {
                const float2 a = w[p], b = w[p + s];
                w[p] = fadd2(a, b);
                w[p + s] = fsub2(a, b);
            }
        }
    }
#pragma unroll
    for (int m = 1; m < 4; m <<= 1) {
        const float sg = (j & m) ? -1.0f : 1.0f;
        const float2 sg2 = make_float2(sg, sg);
#pragma unroll
        for (int p = 0; p < NP; ++p) {
            const float2 other = make_float2(__shfl_xor_sync(0xffffffffu, w[p].x, m),
                                             __shfl_xor_sync(0xffffffffu, w[p].y, m));
            w[p] = ffma2(w[p], sg2, other);
        }
    }
}

// This lane's chunks of `row` (zeros past the end).
template <int D>
__device__ __forceinline__ void load_chunks(const uint4 *__restrict__ x, long row, long rows, int j,
                                            uint4 (&u)[HqShape<D>::CPL]) {
#pragma unroll
    for (int k = 0; k < HqShape<D>::CPL; ++k)
        u[k] = row < rows ? x[row * (D / 8) + 4 * k + j] : make_uint4(0u, 0u, 0u, 0u);
}

// Widens the chunks to float pairs with the signs applied (a flip of each
// bf16 sign bit, `flip` holding the bits per 32-bit word) and transforms
// them when signs are given; the 1/sqrt(d) factor is not applied.
template <int D>
__device__ __forceinline__ void rotate_raw(const uint4 (&u)[HqShape<D>::CPL], const uint32_t (&flip)[HqShape<D>::VPL / 2],
                                          bool use_signs, int j, float2 (&w)[HqShape<D>::VPL / 2]) {
#pragma unroll
    for (int k = 0; k < HqShape<D>::CPL; ++k) {
        const uint32_t q[4] = {u[k].x, u[k].y, u[k].z, u[k].w};
#pragma unroll
        for (int i = 0; i < 4; ++i) w[4 * k + i] = unpack2<true>(q[i] ^ flip[4 * k + i]);
    }
    if (use_signs) hadamard_pairs<D>(w, j);  // all lanes of the warp take part
}

// This lane's sign flips: for the pair of values 8 (4 k + j) + 2 i, + 1, the
// sign bits of the two bf16 halves of a word.
template <int D>
__device__ __forceinline__ void load_flips(const float *__restrict__ signs, int j, uint32_t (&flip)[HqShape<D>::VPL / 2]) {
#pragma unroll
    for (int k = 0; k < HqShape<D>::CPL; ++k)
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int v = 8 * (4 * k + j) + 2 * i;
            flip[4 * k + i] = signs ? ((signs[v] < 0.0f ? 0x8000u : 0u) | (signs[v + 1] < 0.0f ? 0x80000000u : 0u)) : 0u;
        }
}

__global__ void hq_zero_kernel(float *amax) { *amax = 0.0f; }

template <int D>
__global__ void __launch_bounds__(256) hq_amax_kernel(const uint4 *__restrict__ x, const float *__restrict__ signs,
                                                      float *__restrict__ amax, long rows) {
    using S = HqShape<D>;
    constexpr int kU = S::KU;
    const long warp_id = ((long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const long nwarps = ((long)gridDim.x * blockDim.x) >> 5;
    const int lane = threadIdx.x & 31;
    const int j = lane & 3;
    uint32_t flip[S::VPL / 2];
    load_flips<D>(signs, j, flip);
    float m = 0.0f;  // max |v| before the 1/sqrt(d) factor (applied once below: the order is the same)
    // warp-uniform trip count: the shuffles inside need every lane
    for (long base = warp_id * S::RPW * kU; base < rows; base += nwarps * S::RPW * kU) {
        uint4 u[kU][S::CPL];
#pragma unroll
        for (int q = 0; q < kU; ++q) load_chunks<D>(x, base + q * S::RPW + (lane >> 2), rows, j, u[q]);
#pragma unroll
        for (int q = 0; q < kU; ++q) {
            float2 w[S::VPL / 2];
            rotate_raw<D>(u[q], flip, signs != nullptr, j, w);
#pragma unroll
            for (int p = 0; p < S::VPL / 2; ++p) m = fmaxf(m, fmaxf(fabsf(w[p].x), fabsf(w[p].y)));
        }
    }
    if (signs) m *= D == 128 ? 0.08838834764831845f : 0.125f;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
    __shared__ float wmax[8];
    if (lane == 0) wmax[threadIdx.x >> 5] = m;
    __syncthreads();
    if (threadIdx.x == 0) {
        float bm = 0.0f;
        for (int i = 0; i < (int)(blockDim.x >> 5); ++i) bm = fmaxf(bm, wmax[i]);
        // non-negative floats order like their bit patterns
        atomicMax(reinterpret_cast<int *>(amax), __float_as_int(bm));
    }
}

template <int D>
__global__ void __launch_bounds__(256) hq_quant_kernel(const uint4 *__restrict__ x, const float *__restrict__ signs,
                                                       const float *__restrict__ amax, uint2 *__restrict__ x8,
                                                       float *__restrict__ descale, long rows) {
    using S = HqShape<D>;
    constexpr int kU = S::KU;
    const float a = *amax;
    const float inv = a > 0.0f ? 448.0f / a : 1.0f;
    if (blockIdx.x == 0 && threadIdx.x == 0) *descale = a > 0.0f ? a / 448.0f : 1.0f;
    const float c = signs ? (D == 128 ? 0.08838834764831845f : 0.125f) : 1.0f;  // 1/sqrt(d) of the transform
    const float2 c2 = make_float2(c, c), inv2 = make_float2(inv, inv);
    const long warp_id = ((long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const long nwarps = ((long)gridDim.x * blockDim.x) >> 5;
    const int lane = threadIdx.x & 31;
    const int j = lane & 3;
    uint32_t flip[S::VPL / 2];
    load_flips<D>(signs, j, flip);
    for (long base = warp_id * S::RPW * kU; base < rows; base += nwarps * S::RPW * kU) {
        uint4 u[kU][S::CPL];
#pragma unroll
        for (int q = 0; q < kU; ++q) load_chunks<D>(x, base + q * S::RPW + (lane >> 2), rows, j, u[q]);
#pragma unroll
        for (int q = 0; q < kU; ++q) {
            const long row = base + q * S::RPW + (lane >> 2);
            float2 w[S::VPL / 2];
            rotate_raw<D>(u[q], flip, signs != nullptr, j, w);
            if (row < rows) {
#pragma unroll
                for (int k = 0; k < S::CPL; ++k) {
                    float2 t[4];
#pragma unroll
                    for (int i = 0; i < 4; ++i) t[i] = fmul2(fmul2(w[4 * k + i], c2), inv2);
                    const uint32_t lo = cvt_e4m3x2(t[0].x, t[0].y) | (cvt_e4m3x2(t[1].x, t[1].y) << 16);
                    const uint32_t hi = cvt_e4m3x2(t[2].x, t[2].y) | (cvt_e4m3x2(t[3].x, t[3].y) << 16);
                    x8[row * (D / 8) + 4 * k + j] = make_uint2(lo, hi);
                }
            }
        }
    }
}

// ----------------------------------------------------------- FP8 forward
// Two 128-row Q tiles per CTA with ping-ponged softmax warpgroups, as in the
// bf16 forward: warps 0-3 tile A, 4-7 tile B, warp 8 TMA producer, warp 9
// MMA issuer.  Tensor memory: S_A [0,128), S_B [128,256), O_A [256,384),
// O_B [384,512); P (e4m3, 32 columns) overlays the first columns of its own
// S.  MMA order per K/V tile j: O_A += P_A V_j, S_A(j+1), O_B += P_B V_j,
// S_B(j+1), so S_X(j+1) completes after O_X += P_X(j) V_j.

constexpr int kBM = 128, kBN = 128, kD = 128;
constexpr int kThreads = 320;
constexpr int kProducerWarp = 8, kMmaWarp = 9;
constexpr float kRescaleThreshold = 4.0f;  // log2 units
constexpr float kLift = 4.0f;              // P is quantised as 2^(s - m + kLift)

struct Fp8Layout {
    static constexpr int KS = 3, VS = 3;
    static constexpr int TILE = kBM * kD;  // bytes (1 byte per value)
    static constexpr int OFF_Q = 0;        // Q_A, Q_B
    static constexpr int OFF_K = OFF_Q + 2 * TILE;
    static constexpr int OFF_V = OFF_K + KS * TILE;
    static constexpr int OFF_O = OFF_V + VS * TILE;  // bf16 output staging: per tile 2 boxes of 128 x 64
    static constexpr int OTILE = kBM * kD * 2;
    static constexpr int OFF_BAR = OFF_O + 2 * OTILE;
    // q_full, k_full[KS], k_empty[KS], v_full[VS], v_empty[VS], s_full[2],
    // p_full[2], o_final[2], drain
    static constexpr int NBAR = 1 + 2 * KS + 2 * VS + 2 + 2 + 2 + 1;
    static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
    static constexpr int BYTES = OFF_MISC + 16;
    static constexpr int ALLOC = BYTES + 1024;
    static_assert(ALLOC <= 227 * 1024, "shared memory");
};

struct Fp8Params {
    float *lse;
    const float *q_descale, *k_descale, *v_descale;
    unsigned int *status;
    int Hq, Hkv, N, nblk, causal;  // nblk: 256-row blocks per head
    int group, planes;             // CTA order (grid_order.cuh): planes per group, B * Hq
    float scale_log2;
};

constexpr uint32_t kColS = 0, kColO = 256;  // + 128 per tile

__global__ void __launch_bounds__(kThreads, 1)
    fwd_fp8_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                   const Fp8Params p) {
    using L = Fp8Layout;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::OFF_BAR);
    uint64_t *q_full = bars;
    uint64_t *k_full = q_full + 1;
    uint64_t *k_empty = k_full + L::KS;
    uint64_t *v_full = k_empty + L::KS;
    uint64_t *v_empty = v_full + L::VS;
    uint64_t *s_full = v_empty + L::VS;  // [2], one per tile
    uint64_t *p_full = s_full + 2;       // [2]
    uint64_t *o_final = p_full + 2;      // [2]
    uint64_t *drain = o_final + 2;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L::OFF_MISC);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::OFF_MISC + 4);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    // CTA order: planes in L2-sized groups, longest causal blocks first
    int bh, t_lin;
    grid_decode(blockIdx.x, p.planes, p.nblk, p.group, bh, t_lin);
    const int t = p.causal ? (p.nblk - 1 - t_lin) : t_lin;
    const int b = bh / p.Hq;
    const int h = bh - b * p.Hq;
    const int hk = h / (p.Hq / p.Hkv);
    const int q0a = t * 2 * kBM;
    const int nkv_all = (p.N + kBN - 1) / kBN;
    // K/V tiles each Q tile visits; 0 for a tile that lies entirely past N
    const int nA = p.causal ? min(q0a / kBN + 1, nkv_all) : nkv_all;
    const int nB = q0a + kBM >= p.N ? 0 : (p.causal ? min((q0a + kBM) / kBN + 1, nkv_all) : nkv_all);
    const int nmax = max(nA, nB);
    const int kv_plane = b * p.Hkv + hk;
    const int q_plane = b * p.Hq + h;

    if (threadIdx.x == 0) {
        mbar_init(q_full, 1);
        for (int s = 0; s < L::KS; ++s) { mbar_init(&k_full[s], 1); mbar_init(&k_empty[s], 1); }
        for (int s = 0; s < L::VS; ++s) { mbar_init(&v_full[s], 1); mbar_init(&v_empty[s], 1); }
        for (int x = 0; x < 2; ++x) {
            mbar_init(&s_full[x], 1);
            mbar_init(&p_full[x], kBM);
            mbar_init(&o_final[x], 1);
        }
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == kMmaWarp) {
        tmem_alloc(tmem_slot, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == kProducerWarp) {
        // -------------------------------------------------------- TMA producer
        if (lane == 0) {
            prefetch_tmap(&tm_q);
            prefetch_tmap(&tm_k);
            prefetch_tmap(&tm_v);
            const int ntq = nB > 0 ? 2 : 1;
            mbar_arrive_expect_tx(q_full, ntq * L::TILE);
            for (int x = 0; x < ntq; ++x)
                tma_load_3d(smem + L::OFF_Q + x * L::TILE, &tm_q, q_full, 0, q0a + x * kBM, q_plane);
            int nk = 0, nv = 0;
            for (int j = 0; j < nmax; ++j) {
                const int ks = j % L::KS;
                if (j >= L::KS && !mbar_wait(&k_empty[ks], ((j / L::KS) + 1) & 1, abort_flag, p.status, 41)) break;
                mbar_arrive_expect_tx(&k_full[ks], L::TILE);
                tma_load_3d(smem + L::OFF_K + ks * L::TILE, &tm_k, &k_full[ks], 0, j * kBN, kv_plane);
                ++nk;
                const int vs = j % L::VS;
                if (j >= L::VS && !mbar_wait(&v_empty[vs], ((j / L::VS) + 1) & 1, abort_flag, p.status, 42)) break;
                mbar_arrive_expect_tx(&v_full[vs], L::TILE);
                tma_load_3d(smem + L::OFF_V + vs * L::TILE, &tm_v, &v_full[vs], 0, j * kBN, kv_plane);
                ++nv;
            }
            if (*abort_flag) {
                // let copies already in flight land before the CTA exits
                mbar_wait_drain(q_full, 0, 10000000ull);
                for (int u = max(0, nk - L::KS); u < nk; ++u)
                    mbar_wait_drain(&k_full[u % L::KS], (u / L::KS) & 1, 10000000ull);
                for (int u = max(0, nv - L::VS); u < nv; ++u)
                    mbar_wait_drain(&v_full[u % L::VS], (u / L::VS) & 1, 10000000ull);
            }
        }
        __syncwarp();
    } else if (warp == kMmaWarp) {
        // ------------------------------------------------------- MMA issuer
        if (lane == 0) {
            // kind::f8f6f4, e4m3 (format 0) for both operands, fp32 accumulate
            constexpr uint32_t idesc_s = make_idesc(kBM, kBN, 0u, false, false);
            constexpr uint32_t idesc_pv = make_idesc(kBM, kD, 0u, false, true);
            const uint64_t q_desc0 = make_sdesc_sw128(smem_u32(smem + L::OFF_Q), 16, 1024);
            const uint64_t k_desc0 = make_sdesc_sw128(smem_u32(smem + L::OFF_K), 16, 1024);
            const uint64_t v_desc0 = make_sdesc_sw128(smem_u32(smem + L::OFF_V), 0, 1024);
            int k_ready = -1;  // highest K tile whose arrival has been observed

            auto wait_k = [&](int j) -> bool {
                if (j <= k_ready) return true;
                if (!mbar_wait(&k_full[j % L::KS], (j / L::KS) & 1, abort_flag, p.status, 43)) return false;
                tc_fence_after();
                k_ready = j;
                return true;
            };
            // S_x(j) = Q_x K_j^T: both operands K-major e4m3, 32 values = 32
            // bytes per step inside the 128-byte row
            auto issue_s = [&](int x, int j) {
                const uint64_t q_desc = sdesc_advance(q_desc0, x * L::TILE);
                const uint64_t k_desc = sdesc_advance(k_desc0, (j % L::KS) * L::TILE);
#pragma unroll
                for (int kk = 0; kk < kD / 32; ++kk)
                    mma_f8_ss(tmem + kColS + x * 128, sdesc_advance(q_desc, kk * 32), sdesc_advance(k_desc, kk * 32),
                              idesc_s, kk > 0 ? 1u : 0u);
                mma_commit(&s_full[x]);
            };
            // O_x += P_x(j) V_j: A = P from tensor memory (32 keys = 8 columns
            // per step), B = V with the head dim contiguous (MN-major), 32
            // keys = 32 rows of 128 bytes per step
            auto issue_pv = [&](int x, int j) -> bool {
                if (!mbar_wait(&p_full[x], j & 1, abort_flag, p.status, 44)) return false;
                tc_fence_after();
                const uint64_t v_desc = sdesc_advance(v_desc0, (j % L::VS) * L::TILE);
                const uint32_t p_col = tmem + kColS + x * 128;
#pragma unroll
                for (int kk = 0; kk < kBN / 32; ++kk)
                    mma_f8_ts(tmem + kColO + x * 128, p_col + kk * 8, sdesc_advance(v_desc, kk * 32 * 128), idesc_pv,
                              (j > 0 || kk > 0) ? 1u : 0u);
                return true;
            };

            bool ok = mbar_wait(q_full, 0, abort_flag, p.status, 45);
            if (ok) {
                tc_fence_after();
                ok = wait_k(0);
            }
            if (ok) {
                issue_s(0, 0);
                if (nB > 0) issue_s(1, 0);
                mma_commit(&k_empty[0]);
            }
            for (int j = 0; ok && j < nmax; ++j) {
                if (!mbar_wait(&v_full[j % L::VS], (j / L::VS) & 1, abort_flag, p.status, 46)) { ok = false; break; }
                tc_fence_after();
                for (int x = 0; x < 2; ++x) {
                    const int nx = x ? nB : nA;
                    if (j >= nx) continue;
                    if (!issue_pv(x, j)) { ok = false; break; }
                    if (j + 1 < nx) {
                        // S_x(j+1) overwrites P_x(j), which the MMAs just issued read first
                        if (!wait_k(j + 1)) { ok = false; break; }
                        issue_s(x, j + 1);
                    } else {
                        mma_commit(&o_final[x]);
                    }
                }
                if (!ok) break;
                mma_commit(&v_empty[j % L::VS]);
                if (j + 1 < nmax) mma_commit(&k_empty[(j + 1) % L::KS]);
            }
            // every MMA issued above has completed once `drain` flips
            mma_commit(drain);
            mbar_wait_drain(drain, 0, 100000000ull);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------ softmax + epilogue
        const int x = warp >> 2;  // tile
        const int quarter = warp & 3;
        const int row = quarter * 32 + lane;  // query row within the tile == TMEM lane
        const uint32_t lane_base = tmem + ((uint32_t)(quarter * 32) << 16);
        const uint32_t col_s = kColS + x * 128, col_o = kColO + x * 128;
        const int q0 = q0a + x * kBM;
        const int nx = x ? nB : nA;
        const float sl2 = p.scale_log2 * (*p.q_descale) * (*p.k_descale);
        float m_ref = -INFINITY;
        float l_sum = 0.0f;    // sum of the quantised P (lifted): normalises O
        float l_exact = 0.0f;  // sum of the unquantised P (lifted): gives L
        bool ok = true;

        for (int j = 0; ok && j < nx; ++j) {
            // every lane waits, then the warp votes: the tcgen05.ld/st below
            // are warp-collective (.sync.aligned) and need all 32 lanes
            const bool got_s = mbar_wait(&s_full[x], j & 1, abort_flag, p.status, 47);
            if (!__all_sync(0xffffffffu, got_s)) { ok = false; break; }
            tc_fence_after();
            uint32_t s[128];
            const uint32_t s_addr = lane_base + col_s;
            tmem_ld_x32(s_addr + 0, s + 0);
            tmem_ld_x32(s_addr + 32, s + 32);
            tmem_ld_x32(s_addr + 64, s + 64);
            tmem_ld_x32(s_addr + 96, s + 96);
            tmem_ld_wait_x32(s + 0);
            tmem_ld_wait_x32(s + 32);
            tmem_ld_wait_x32(s + 64);
            tmem_ld_wait_x32(s + 96);

            const int kv0 = j * kBN;
            const bool need_mask = (kv0 + kBN > p.N) || (p.causal && kv0 + kBN - 1 > q0);
            if (need_mask) {
                const int lim = p.causal ? min(p.N, q0 + row + 1) : p.N;
#pragma unroll
                for (int c = 0; c < 128; ++c)
                    if (kv0 + c >= lim) s[c] = __float_as_uint(-INFINITY);
            }
            // four chains of three-input maxima: two new scores per instruction
            float mx0 = -INFINITY, mx1 = -INFINITY, mx2 = -INFINITY, mx3 = -INFINITY;
#pragma unroll
            for (int c = 0; c < 128; c += 8) {
                mx0 = fmax3(mx0, __uint_as_float(s[c]), __uint_as_float(s[c + 1]));
                mx1 = fmax3(mx1, __uint_as_float(s[c + 2]), __uint_as_float(s[c + 3]));
                mx2 = fmax3(mx2, __uint_as_float(s[c + 4]), __uint_as_float(s[c + 5]));
                mx3 = fmax3(mx3, __uint_as_float(s[c + 6]), __uint_as_float(s[c + 7]));
            }
            const float mx = fmaxf(fmaxf(mx0, mx1), fmaxf(mx2, mx3)) * sl2;
            float alpha = 1.0f;
            bool rescale = false;
            if (mx > m_ref + kRescaleThreshold) {
                alpha = ex2_approx(m_ref - mx);
                l_sum *= alpha;
                l_exact *= alpha;
                m_ref = mx;
                rescale = true;
            }
            __syncwarp();  // reconverge after the per-row branches above
            const float2 bias = make_float2(kLift - m_ref, kLift - m_ref);
            const float2 sl2x2 = make_float2(sl2, sl2);
            float2 le01 = make_float2(0.f, 0.f), le23 = le01;
            // the sum of the quantised P is accumulated in fp16 pairs over 32
            // scores (each half adds 8 values of at most 256: no overflow, but
            // every add rounds to fp16's 11-bit significand, about 2^-11
            // relative) and then widened, which costs one conversion and one
            // add per two scores instead of widening every value
            float lr = 0.0f;
#pragma unroll
            for (int hh = 0; hh < 4; ++hh) {
                uint32_t pk[8];
                uint32_t hacc0 = 0u, hacc1 = 0u;
#pragma unroll
                for (int c = 32 * hh; c < 32 * hh + 32; c += 4) {
                    const float2 x01 =
                        ffma2(make_float2(__uint_as_float(s[c]), __uint_as_float(s[c + 1])), sl2x2, bias);
                    const float2 x23 =
                        ffma2(make_float2(__uint_as_float(s[c + 2]), __uint_as_float(s[c + 3])), sl2x2, bias);
                    const float p0 = ex2_approx(x01.x);
                    const float p1 = ex2_approx(x01.y);
                    const float p2 = ex2_approx(x23.x);
                    const float p3 = ex2_approx(x23.y);
                    const uint32_t w01 = cvt_e4m3x2(p0, p1);
                    const uint32_t w23 = cvt_e4m3x2(p2, p3);
                    pk[(c - 32 * hh) / 4] = w01 | (w23 << 16);
                    hacc0 = hadd2_u32(hacc0, e4m3x2_to_h2(w01));
                    hacc1 = hadd2_u32(hacc1, e4m3x2_to_h2(w23));
                    le01 = fadd2(le01, make_float2(p0, p1));
                    le23 = fadd2(le23, make_float2(p2, p3));
                }
                const float2 f0 = unpack2<false>(hacc0);
                const float2 f1 = unpack2<false>(hacc1);
                lr += (f0.x + f0.y) + (f1.x + f1.y);
                // P of keys 32 hh .. + 31 -> columns 8 hh .. + 7 of this row's S,
                // all of which have been read
                tmem_st_x8(lane_base + col_s + 8 * hh, pk);
            }
            l_sum += lr;
            l_exact += (le01.x + le01.y) + (le23.x + le23.y);
            // O_x already holds P_x(0..j-1) V (S_x(j) was issued after the last
            // P.V of this tile), and P_x(j) V is issued only after p_full;
            // warp-uniform branch, lanes that keep their max use alpha = 1
            if (j >= 1 && __any_sync(0xffffffffu, rescale)) {
                // one tensor-memory round trip: the S registers are free again
                uint32_t o[kD];
#pragma unroll
                for (int c0 = 0; c0 < kD; c0 += 32) tmem_ld_x32(lane_base + col_o + c0, o + c0);
#pragma unroll
                for (int c0 = 0; c0 < kD; c0 += 32) tmem_ld_wait_x32(o + c0);
#pragma unroll
                for (int c = 0; c < kD; c += 2) {
                    const float2 r = fmul2(make_float2(__uint_as_float(o[c]), __uint_as_float(o[c + 1])),
                                           make_float2(alpha, alpha));
                    o[c] = __float_as_uint(r.x);
                    o[c + 1] = __float_as_uint(r.y);
                }
#pragma unroll
                for (int c0 = 0; c0 < kD; c0 += 32) tmem_st_x32(lane_base + col_o + c0, o + c0);
            }
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(&p_full[x]);
        }

        if (nx > 0) {  // uniform across the warpgroup
            if (ok) ok = mbar_wait(&o_final[x], 0, abort_flag, p.status, 49);
            __syncwarp();
            // uniform decision across the tile's 128 threads (the epilogue has a
            // named barrier that all of them must reach)
            ok = named_bar_and(1 + x, kBM, ok);
            if (ok) {
                tc_fence_after();
                // O = v_descale * O~ / l, bf16, staged in the 128-byte-swizzled
                // layout of two 64-column output boxes
                const float f = (*p.v_descale) / l_sum;
                uint8_t *stage = smem + L::OFF_O + x * L::OTILE;
#pragma unroll 1
                for (int c0 = 0; c0 < kD; c0 += 32) {
                    uint32_t o[32];
                    tmem_ld_x32(lane_base + col_o + c0, o);
                    tmem_ld_wait_x32(o);
                    uint32_t w[16];
#pragma unroll
                    for (int c = 0; c < 16; ++c)
                        w[c] = pack_bf16x2(__uint_as_float(o[2 * c]) * f, __uint_as_float(o[2 * c + 1]) * f);
                    uint8_t *rowp = stage + (c0 >> 6) * (kBM * 128) + row * 128;
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const int chunk = ((c0 & 63) >> 3) + q;
                        *reinterpret_cast<uint4 *>(rowp + ((chunk ^ (row & 7)) << 4)) =
                            make_uint4(w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]);
                    }
                }
                fence_proxy_async_smem();
                named_bar_sync(1 + x, kBM);
                if (row == 0) {
                    for (int bx = 0; bx < 2; ++bx)
                        tma_store_3d(&tm_o, stage + bx * (kBM * 128), bx * 64, q0, q_plane);
                    bulk_commit();
                    bulk_wait_read_all();
                }
                if (q0 + row < p.N)
                    p.lse[(size_t)q_plane * p.N + q0 + row] =
                        (m_ref + log2f(l_exact) - kLift) * 0.69314718055994530942f;
            }
        }
        __syncwarp();
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

int stream_blocks() {
    int dev = 0, sms = 152;
    if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    return sms * 8;
}

template <int D>
cudaError_t launch_hq_t(const QuantArgs &a, cudaStream_t st) {
    const int nb = stream_blocks();
    hq_zero_kernel<<<1, 1, 0, st>>>(a.amax);
    hq_amax_kernel<D><<<nb, 256, 0, st>>>(static_cast<const uint4 *>(a.x), a.signs, a.amax, a.rows);
    hq_quant_kernel<D><<<nb, 256, 0, st>>>(static_cast<const uint4 *>(a.x), a.signs, a.amax,
                                           static_cast<uint2 *>(a.x8), a.descale, a.rows);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_hadamard_quant(const QuantArgs &a, cudaStream_t st) {
    if (a.d == 128) return launch_hq_t<128>(a, st);
    if (a.d == 64) return launch_hq_t<64>(a, st);
    return cudaErrorInvalidValue;
}

cudaError_t launch_fwd_fp8(const Fp8FwdArgs &a, cudaStream_t st) {
    if (a.d != kD) return cudaErrorInvalidValue;
    using L = Fp8Layout;
    CUtensorMap tq, tk, tv, to;
    const uint64_t N = a.N;
    if (!make_tmap_3d(&tq, a.q8, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, kD, N, (uint64_t)a.B * a.Hq, 128, kBM,
                      CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_tmap_3d(&tk, a.k8, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, kD, N, (uint64_t)a.B * a.Hkv, 128, kBN,
                      CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_tmap_3d(&tv, a.v8, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, kD, N, (uint64_t)a.B * a.Hkv, 128, kBN,
                      CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_tmap_3d(&to, a.o, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, kD, N, (uint64_t)a.B * a.Hq, 64, kBM,
                      CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(fwd_fp8_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, L::ALLOC);
    if (e != cudaSuccess) return e;
    Fp8Params p;
    p.lse = a.lse;
    p.q_descale = a.q_descale;
    p.k_descale = a.k_descale;
    p.v_descale = a.v_descale;
    p.status = device_status_ptr();
    p.Hq = a.Hq;
    p.Hkv = a.Hkv;
    p.N = a.N;
    p.nblk = (a.N + 2 * kBM - 1) / (2 * kBM);
    {
        int dev = 0, sms = 0;
        if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
        if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
        p.planes = a.B * a.Hq;
        p.group = grid_group_planes(p.planes, p.nblk, sms);
    }
    p.causal = a.causal;
    p.scale_log2 = a.scale * 1.4426950408889634f;
    const long long grid = (long long)p.nblk * a.B * a.Hq;
    fwd_fp8_kernel<<<dim3((unsigned)grid), dim3(kThreads), L::ALLOC, st>>>(tq, tk, tv, to, p);
    return cudaGetLastError();
}

}  // namespace fa
