// fa_fwd.cu -- FlashAttention-2 forward for sm_103a (bf16 / fp16, d = 64, 128).
//
// Algorithm ("6.2 FlashAttention V2 chi tiet", section 6.1; blog.csdn.net
// FlashAttention-2 article, 3.1.1): one CTA per (Q tile of 128 rows, query
// head, batch); the Q tile is loaded once and stays in shared memory while the
// CTA walks the K/V tiles; the running row max m and row sum l are updated per
// tile, the output is accumulated unnormalised and divided by l once at the
// end, and only L = m + log l is stored.  Causal: tiles above the diagonal are
// never visited (the loop stops at the diagonal tile) and only the diagonal
// tile is masked element-wise (section 5.3).
//
// GB300 realisation (warp-specialised, one CTA per SM):
//   warp 4  lane 0   TMA producer for Q (once) and the K ring
//   warp 6  lane 0   TMA producer for the V ring
//   warp 5  lane 0   tcgen05 MMA issuer; warp 5 also owns the TMEM allocation
//   warps 0-3        softmax: thread t owns query row t = TMEM lane t, so a
//                    row's max and sum never leave one thread (the page's
//                    split of rows across warps, section 4.2, taken to its
//                    limit), then the epilogue.
// Tensor memory (512 columns x 128 lanes, fp32):
//   [0,128) S buffer 0   [128,256) S buffer 1   [256,256+d) O accumulator
//   [384,384+d/2) Q (16-bit pairs, the A operand of S = Q K^T, copied once)
// P (16-bit pairs) overwrites the first 64 columns of its own S buffer (each
// softmax thread writes only its own lane, after reading the whole row) and is
// the A operand of the P.V MMA.  With Q and P read from tensor memory only K
// and V occupy the shared-memory operand path (128 bytes / cycle).
// Pipeline per K/V tile j: MMA S_j = Q K_j^T -> softmax_j (P_j, row stats)
// -> MMA O += P_j V_j.  S is double-buffered so S_{j+1} runs on the tensor
// cores while softmax_j runs, and softmax_{j+1} overlaps O += P_j V_j.
//
// Exact lazy rescaling: the reference max m_ref of a row moves only when the
// tile max exceeds it by more than 8 (log2 units); then O and l are rescaled
// by 2^(m_ref_old - m_ref_new) once.  Between moves P = 2^(s - m_ref) <= 2^8,
// and because O~ and l always share the same m_ref the final O~ / l is the
// same quotient as with the page's per-tile update.
#include "host_util.h"
#include "ptx.cuh"

namespace fa {

namespace {

constexpr int kBM = 128;      // query rows per CTA (TMEM lanes)
constexpr int kBN = 128;      // keys per K/V tile
constexpr int kThreads = 224; // 7 warps
constexpr float kRescaleThreshold = 8.0f;

template <int D>
struct FwdLayout {
    static constexpr int KS = 3;  // K ring depth
    static constexpr int VS = 2;  // V ring depth
    static constexpr int NBOX = D / 64;           // 64-column (128-byte) boxes
    static constexpr int TILE_Q = kBM * D * 2;    // bytes
    static constexpr int TILE_KV = kBN * D * 2;
    static constexpr int OFF_Q = 0;
    static constexpr int OFF_K = OFF_Q + TILE_Q;
    static constexpr int OFF_V = OFF_K + KS * TILE_KV;
    static constexpr int OFF_BAR = OFF_V + VS * TILE_KV;
    // q_full, q_tmem, k_full[KS], k_empty[KS], v_full[VS], v_empty[VS],
    // s_full[2], p_full[2], o_done, drain
    static constexpr int NBAR = 2 + 2 * KS + 2 * VS + 2 + 2 + 1 + 1;
    static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
    static constexpr int BYTES = OFF_MISC + 16;
    static constexpr int ALLOC = BYTES + 1024;  // room to align the base to 1024
};

struct FwdParams {
    float *lse;
    unsigned int *status;
    int Hq, Hkv, N, nqt, causal;
    float scale_log2;  // scale * log2(e)
};

constexpr uint32_t kColS = 0, kColO = 256, kColQ = 384;

template <int D, bool BF16>
__global__ void __launch_bounds__(kThreads, 1)
    fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
               const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
               const FwdParams p) {
    using L = FwdLayout<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::OFF_BAR);
    uint64_t *q_full = bars;
    uint64_t *q_tmem = bars + 1;
    uint64_t *k_full = q_tmem + 1;
    uint64_t *k_empty = k_full + L::KS;
    uint64_t *v_full = k_empty + L::KS;
    uint64_t *v_empty = v_full + L::VS;
    uint64_t *s_full = v_empty + L::VS;
    uint64_t *p_full = s_full + 2;
    uint64_t *o_done = p_full + 2;
    uint64_t *drain = o_done + 1;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L::OFF_MISC);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::OFF_MISC + 4);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    // Tile schedule: consecutive CTAs share a head (K/V stay hot in L2);
    // within a head, causal tiles go longest first.
    const int bh = blockIdx.x / p.nqt;
    const int qt_lin = blockIdx.x - bh * p.nqt;
    const int qt = p.causal ? (p.nqt - 1 - qt_lin) : qt_lin;
    const int b = bh / p.Hq;
    const int h = bh - b * p.Hq;
    const int hk = h / (p.Hq / p.Hkv);
    const int q0 = qt * kBM;
    const int nkv_all = (p.N + kBN - 1) / kBN;
    const int nkv = p.causal ? min(qt + 1, nkv_all) : nkv_all;
    const int kv_plane = b * p.Hkv + hk;
    const int q_plane = b * p.Hq + h;

    if (threadIdx.x == 0) {
        mbar_init(q_full, 1);
        mbar_init(q_tmem, kBM);
        for (int s = 0; s < L::KS; ++s) { mbar_init(&k_full[s], 1); mbar_init(&k_empty[s], 1); }
        for (int s = 0; s < L::VS; ++s) { mbar_init(&v_full[s], 1); mbar_init(&v_empty[s], 1); }
        for (int s = 0; s < 2; ++s) { mbar_init(&s_full[s], 1); mbar_init(&p_full[s], kBM); }
        mbar_init(o_done, 1);
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 5) {
        tmem_alloc(tmem_slot, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 4) {
        // ---------------------------------------------------- Q + K producer
        if (lane == 0) {
            prefetch_tmap(&tm_q);
            prefetch_tmap(&tm_k);
            mbar_arrive_expect_tx(q_full, L::TILE_Q);
            for (int bx = 0; bx < L::NBOX; ++bx)
                tma_load_3d(smem + L::OFF_Q + bx * kBM * 128, &tm_q, q_full, bx * 64, q0, q_plane);
            int j = 0;
            for (; j < nkv; ++j) {
                const int s = j % L::KS;
                if (j >= L::KS && !mbar_wait(&k_empty[s], ((j / L::KS) + 1) & 1, abort_flag, p.status, 1)) break;
                mbar_arrive_expect_tx(&k_full[s], L::TILE_KV);
                uint8_t *dst = smem + L::OFF_K + s * L::TILE_KV;
                for (int bx = 0; bx < L::NBOX; ++bx)
                    tma_load_3d(dst + bx * kBN * 128, &tm_k, &k_full[s], bx * 64, j * kBN, kv_plane);
            }
            if (*abort_flag) {
                // let copies already in flight land before the CTA exits
                for (int t = max(0, j - L::KS); t < j; ++t)
                    mbar_wait_drain(&k_full[t % L::KS], (t / L::KS) & 1, 10000000ull);
                mbar_wait_drain(q_full, 0, 10000000ull);
            }
        }
        __syncwarp();
    } else if (warp == 6) {
        // -------------------------------------------------------- V producer
        if (lane == 0) {
            prefetch_tmap(&tm_v);
            int j = 0;
            for (; j < nkv; ++j) {
                const int s = j % L::VS;
                if (j >= L::VS && !mbar_wait(&v_empty[s], ((j / L::VS) + 1) & 1, abort_flag, p.status, 2)) break;
                mbar_arrive_expect_tx(&v_full[s], L::TILE_KV);
                uint8_t *dst = smem + L::OFF_V + s * L::TILE_KV;
                for (int bx = 0; bx < L::NBOX; ++bx)
                    tma_load_3d(dst + bx * kBN * 128, &tm_v, &v_full[s], bx * 64, j * kBN, kv_plane);
            }
            if (*abort_flag) {
                for (int t = max(0, j - L::VS); t < j; ++t)
                    mbar_wait_drain(&v_full[t % L::VS], (t / L::VS) & 1, 10000000ull);
            }
        }
        __syncwarp();
    } else if (warp == 5) {
        // ------------------------------------------------------- MMA issuer
        if (lane == 0) {
            constexpr uint32_t fmt = BF16 ? 1u : 0u;
            constexpr uint32_t idesc_s = make_idesc(kBM, kBN, fmt, false, false);
            constexpr uint32_t idesc_pv = make_idesc(kBM, D, fmt, false, true);
            // one descriptor per operand tile; steps are derived by sdesc_advance
            const uint64_t k_desc0 = make_sdesc_sw128(smem_u32(smem + L::OFF_K), 16, 1024);
            const uint64_t v_desc0 = make_sdesc_sw128(smem_u32(smem + L::OFF_V), kBN * 128, 1024);
            // Q is in tensor memory once the softmax warps have copied it
            bool ok = mbar_wait(q_tmem, 0, abort_flag, p.status, 3);
            tc_fence_after();

            auto issue_pv = [&](int t) -> bool {
                const int pb = t & 1;
                if (!mbar_wait(&p_full[pb], (t >> 1) & 1, abort_flag, p.status, 4)) return false;
                const int vs = t % L::VS;
                if (!mbar_wait(&v_full[vs], (t / L::VS) & 1, abort_flag, p.status, 5)) return false;
                tc_fence_after();
                const uint64_t v_desc = sdesc_advance(v_desc0, vs * L::TILE_KV);
                const uint32_t p_col = tmem + kColS + pb * kBN;  // P overlays its S buffer
                // B = V (N = d contiguous: MN-major); 16 keys = 16 rows of 128 B
                mma_f16_ts(tmem + kColO, p_col, v_desc, idesc_pv, t > 0 ? 1u : 0u);
#pragma unroll
                for (int kk = 1; kk < kBN / 16; ++kk)
                    mma_f16_ts(tmem + kColO, p_col + kk * 8, sdesc_advance(v_desc, kk * 16 * 128), idesc_pv, 1u);
                mma_commit(o_done);
                mma_commit(&v_empty[vs]);
                return true;
            };

            for (int j = 0; ok && j < nkv; ++j) {
                const int ks = j % L::KS;
                if (!mbar_wait(&k_full[ks], (j / L::KS) & 1, abort_flag, p.status, 6)) { ok = false; break; }
                tc_fence_after();
                const uint64_t k_desc = sdesc_advance(k_desc0, ks * L::TILE_KV);
                const uint32_t s_col = tmem + kColS + (j & 1) * kBN;
                // A = Q from tensor memory (16 head-dim values = 8 columns per
                // step), B = K (K-major, 32 bytes per step inside a 128-byte row)
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t off = (kk >> 2) * (kBN * 128) + (kk & 3) * 32;
                    mma_f16_ts(s_col, tmem + kColQ + kk * 8, sdesc_advance(k_desc, off), idesc_s, kk > 0 ? 1u : 0u);
                }
                mma_commit(&s_full[j & 1]);
                mma_commit(&k_empty[ks]);
                if (j >= 1 && !issue_pv(j - 1)) { ok = false; break; }
            }
            if (ok && nkv > 0) issue_pv(nkv - 1);
            // every MMA issued above has completed once `drain` flips
            mma_commit(drain);
            mbar_wait_drain(drain, 0, 100000000ull);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------ softmax + epilogue
        const int row = threadIdx.x;  // 0..127 == TMEM lane
        const uint32_t lane_base = tmem + ((uint32_t)(warp * 32) << 16);
        const float sl2 = p.scale_log2;
        float m_ref = -INFINITY;
        float l_sum = 0.0f;    // sum of the rounded P fed to the MMA: normalises O
        float l_exact = 0.0f;  // sum of the unrounded P: gives L
        bool ok = true;
        uint32_t s[128];

        {
            // copy this row of Q from the swizzled shared tile into tensor memory
            const bool got_q = mbar_wait(q_full, 0, abort_flag, p.status, 10);
            ok = __all_sync(0xffffffffu, got_q);
            if (ok) {
                uint32_t qv[D / 2];
#pragma unroll
                for (int bx = 0; bx < L::NBOX; ++bx)
#pragma unroll
                    for (int k = 0; k < 8; ++k) {
                        const uint4 u = *reinterpret_cast<const uint4 *>(smem + L::OFF_Q + bx * kBM * 128 + row * 128 +
                                                                         ((k ^ (row & 7)) << 4));
                        qv[bx * 32 + k * 4 + 0] = u.x;
                        qv[bx * 32 + k * 4 + 1] = u.y;
                        qv[bx * 32 + k * 4 + 2] = u.z;
                        qv[bx * 32 + k * 4 + 3] = u.w;
                    }
#pragma unroll
                for (int c0 = 0; c0 < D / 2; c0 += 32) tmem_st_x32(lane_base + kColQ + c0, qv + c0);
                tmem_st_wait();
                tc_fence_before();
                mbar_arrive(q_tmem);
            }
        }

        for (int j = 0; ok && j < nkv; ++j) {
            const int sb = j & 1;
            // every lane waits, then the warp votes: the tcgen05.ld/st below
            // are warp-collective (.sync.aligned) and need all 32 lanes
            const bool got_s = mbar_wait(&s_full[sb], (j >> 1) & 1, abort_flag, p.status, 7);
            if (!__all_sync(0xffffffffu, got_s)) { ok = false; break; }
            tc_fence_after();
            const uint32_t s_addr = lane_base + kColS + sb * kBN;
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
                const int lim = p.causal ? min(p.N, q0 + row + 1) : p.N;  // visible: col < lim
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
                alpha = ex2_approx(m_ref - mx);  // 0 on the first tile (m_ref = -inf)
                l_sum *= alpha;
                l_exact *= alpha;
                m_ref = mx;
                rescale = true;
            }
            const float2 neg_m = make_float2(-m_ref, -m_ref);
            const float2 sl2x2 = make_float2(sl2, sl2);
            float2 lr01 = make_float2(0.f, 0.f), lr23 = lr01, le01 = lr01, le23 = lr01;
            uint32_t pk[64];
#pragma unroll
            for (int c = 0; c < 128; c += 4) {
                const float2 x01 = ffma2(make_float2(__uint_as_float(s[c]), __uint_as_float(s[c + 1])), sl2x2, neg_m);
                const float2 x23 =
                    ffma2(make_float2(__uint_as_float(s[c + 2]), __uint_as_float(s[c + 3])), sl2x2, neg_m);
                const float p0 = ex2_approx(x01.x);
                const float p1 = ex2_approx(x01.y);
                const float p2 = ex2_approx(x23.x);
                const float p3 = ex2_approx(x23.y);
                // l sums the rounded P that the MMA consumes, so O~ / l is an
                // exactly normalised mix of V rows even when one term dominates
                if constexpr (BF16) {
                    pk[c / 2] = pack_bf16x2(p0, p1);
                    pk[c / 2 + 1] = pack_bf16x2(p2, p3);
                } else {
                    pk[c / 2] = pack_f16x2(p0, p1);
                    pk[c / 2 + 1] = pack_f16x2(p2, p3);
                }
                lr01 = fadd2(lr01, unpack2<BF16>(pk[c / 2]));
                lr23 = fadd2(lr23, unpack2<BF16>(pk[c / 2 + 1]));
                le01 = fadd2(le01, make_float2(p0, p1));
                le23 = fadd2(le23, make_float2(p2, p3));
            }
            l_sum += (lr01.x + lr01.y) + (lr23.x + lr23.y);
            l_exact += (le01.x + le01.y) + (le23.x + le23.y);
            __syncwarp();  // reconverge after the per-row branches above
            const uint32_t p_addr = lane_base + kColS + sb * kBN;  // P overlays the S row just read
            tmem_st_x32(p_addr, pk);
            tmem_st_x32(p_addr + 32, pk + 32);

            if (j >= 1) {
                // O holds P_0..P_{j-1} contributions once PV_{j-1} completes
                const bool got_o = mbar_wait(o_done, (j - 1) & 1, abort_flag, p.status, 8);
                if (!__all_sync(0xffffffffu, got_o)) { ok = false; break; }
                // warp-uniform branch; lanes that keep their max use alpha = 1
                if (__any_sync(0xffffffffu, rescale)) {
                    tc_fence_after();
#pragma unroll 1
                    for (int c0 = 0; c0 < D; c0 += 32) {
                        uint32_t o[32];
                        tmem_ld_x32(lane_base + kColO + c0, o);
                        tmem_ld_wait_x32(o);
#pragma unroll
                        for (int c = 0; c < 32; ++c) o[c] = __float_as_uint(__uint_as_float(o[c]) * alpha);
                        tmem_st_x32(lane_base + kColO + c0, o);
                    }
                }
            }
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(&p_full[sb]);
        }

        if (ok && nkv > 0) ok = mbar_wait(o_done, (nkv - 1) & 1, abort_flag, p.status, 9);
        __syncwarp();
        // uniform decision across the 128 softmax threads (the epilogue has a
        // named barrier that all of them must reach)
        ok = named_bar_and(1, kBM, ok);
        if (ok) {
            tc_fence_after();
            // Epilogue: O = O~ / l, staged through the (now idle) Q buffer in
            // the 128-byte-swizzled layout of the output TMA box.
            const float inv_l = 1.0f / l_sum;
            uint8_t *stage = smem + L::OFF_Q;
#pragma unroll 1
            for (int c0 = 0; c0 < D; c0 += 32) {
                uint32_t o[32];
                tmem_ld_x32(lane_base + kColO + c0, o);
                tmem_ld_wait_x32(o);
                uint32_t w[16];
#pragma unroll
                for (int c = 0; c < 16; ++c) {
                    const float a = __uint_as_float(o[2 * c]) * inv_l;
                    const float bb = __uint_as_float(o[2 * c + 1]) * inv_l;
                    w[c] = BF16 ? pack_bf16x2(a, bb) : pack_f16x2(a, bb);
                }
                const int box = c0 >> 6;
                uint8_t *rowp = stage + box * (kBM * 128) + row * 128;
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const int chunk = ((c0 & 63) >> 3) + q;
                    uint4 val = make_uint4(w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]);
                    *reinterpret_cast<uint4 *>(rowp + ((chunk ^ (row & 7)) << 4)) = val;
                }
            }
            fence_proxy_async_smem();
            named_bar_sync(1, kBM);
            if (row == 0) {
                for (int bx = 0; bx < L::NBOX; ++bx)
                    tma_store_3d(&tm_o, stage + bx * (kBM * 128), bx * 64, q0, q_plane);
                bulk_commit();
                bulk_wait_read_all();
            }
            if (q0 + row < p.N)
                p.lse[(size_t)q_plane * p.N + q0 + row] = (m_ref + log2f(l_exact)) * 0.69314718055994530942f;
        }
        __syncwarp();
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 5) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

template <int D, bool BF16>
cudaError_t launch_fwd_t(const FwdArgs &a, cudaStream_t st) {
    using L = FwdLayout<D>;
    const CUtensorMapDataType dt = BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    CUtensorMap tq, tk, tv, to;
    const uint64_t N = a.N;
    if (!make_tmap_3d(&tq, a.q, dt, 2, D, N, (uint64_t)a.B * a.Hq, 64, kBM, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_tmap_3d(&tk, a.k, dt, 2, D, N, (uint64_t)a.B * a.Hkv, 64, kBN, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_tmap_3d(&tv, a.v, dt, 2, D, N, (uint64_t)a.B * a.Hkv, 64, kBN, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_tmap_3d(&to, a.o, dt, 2, D, N, (uint64_t)a.B * a.Hq, 64, kBM, CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(fwd_kernel<D, BF16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         L::ALLOC);
    if (e != cudaSuccess) return e;
    FwdParams p;
    p.lse = a.lse;
    p.status = device_status_ptr();
    p.Hq = a.Hq;
    p.Hkv = a.Hkv;
    p.N = a.N;
    p.nqt = (a.N + kBM - 1) / kBM;
    p.causal = a.causal;
    p.scale_log2 = a.scale * 1.4426950408889634f;
    const long long grid = (long long)p.nqt * a.B * a.Hq;
    fwd_kernel<D, BF16><<<dim3((unsigned)grid), dim3(kThreads), L::ALLOC, st>>>(tq, tk, tv, to, p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd(const FwdArgs &a, cudaStream_t st) {
    if (a.d == 128) return a.bf16 ? launch_fwd_t<128, true>(a, st) : launch_fwd_t<128, false>(a, st);
    if (a.d == 64) return a.bf16 ? launch_fwd_t<64, true>(a, st) : launch_fwd_t<64, false>(a, st);
    return cudaErrorInvalidValue;
}

}  // namespace fa
