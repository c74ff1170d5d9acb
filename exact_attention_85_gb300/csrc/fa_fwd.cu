// fa_fwd.cu -- FlashAttention-2 forward for sm_103a (bf16 / fp16, d = 64, 128).
//
// Algorithm ("6.2 FlashAttention V2 chi tiet", section 6.1; blog.csdn.net
// FlashAttention-2 article, 3.1.1): every 128-row Q tile is loaded once and
// stays on chip while the K/V tiles stream past; the running row max m and
// row sum l are updated per tile, the output is accumulated unnormalised and
// divided by l once at the end, and only L = m + log l is stored.  Causal:
// tiles above the diagonal are never visited (the loop stops at the diagonal
// tile) and only the diagonal tile is masked element-wise (section 5.3).
//
// GB300 realisation: one CTA per SM owns TWO Q tiles (A = rows 0-127,
// B = rows 128-255 of a 256-row block) of one (head, batch), and both walk the
// same K/V stream, so each K/V tile is read once for 256 query rows.  The two
// tiles' softmax warpgroups take turns on the tensor cores: while one
// warpgroup turns S into P, the tensor cores run the other tile's
// P.V and next S (the Blackwell form of the ping-pong the FA3 summary
// describes for two warpgroups).
//   warps 0-3  softmax + epilogue of tile A (thread = query row = TMEM lane)
//   warps 4-7  softmax + epilogue of tile B
//   warp 8     TMA producer (Q once, K ring, V ring)
//   warp 9     tcgen05 MMA issuer; owns the TMEM allocation
// Tensor memory (512 columns x 128 lanes, fp32):
//   [0,128) S_A   [128,256) S_B   [256,256+d) O_A   [384,384+d) O_B
// P (16-bit pairs) overwrites the first 64 columns of its own S (each softmax
// thread writes only its own lane, after reading the whole row) and is the A
// operand of the P.V MMA.  MMA order per K/V tile j:
//   O_A += P_A(j) V_j,  S_A(j+1) = Q_A K_{j+1}^T,  O_B += P_B(j) V_j,  S_B(j+1)
// so S_X(j+1) completes only after O_X += P_X(j) V_j, and a softmax thread
// that needs to rescale O_X may do so as soon as it has seen S_X(j+1).
//
// Exact lazy rescaling: the reference max m_ref of a row moves only when the
// tile max exceeds it by more than 8 (log2 units); then O and l are rescaled
// by 2^(m_ref_old - m_ref_new) once.  Between moves P = 2^(s - m_ref) <= 2^8,
// and because O~ and l always share the same m_ref the final O~ / l is the
// same quotient as with the page's per-tile update.
#include "grid_order.cuh"
#include "host_util.h"
#include "ptx.cuh"

namespace fa {

namespace {

constexpr int kBM = 128;       // query rows per Q tile (TMEM lanes)
constexpr int kBN = 128;       // keys per K/V tile
constexpr int kThreads = 320;  // 10 warps
constexpr int kProducerWarp = 8, kMmaWarp = 9;
constexpr float kRescaleThreshold = 8.0f;

template <int D>
struct FwdLayout {
    static constexpr int KS = D == 128 ? 3 : 4;  // K ring depth
    static constexpr int VS = D == 128 ? 2 : 4;  // V ring depth
    static constexpr int NBOX = D / 64;          // 64-column (128-byte) boxes
    static constexpr int TILE = 128 * D * 2;     // one 128-row tile, bytes
    static constexpr int BOX = 128 * 128;        // one 64-column box of a tile
    static constexpr int OFF_Q = 0;              // Q_A, then Q_B
    static constexpr int OFF_K = OFF_Q + 2 * TILE;
    static constexpr int OFF_V = OFF_K + KS * TILE;
    static constexpr int OFF_BAR = OFF_V + VS * TILE;
    // q_full, k_full[KS], k_empty[KS], v_full[VS], v_empty[VS], s_full[2],
    // p_full[2], o_final[2], drain
    static constexpr int NBAR = 1 + 2 * KS + 2 * VS + 2 + 2 + 2 + 1;
    static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
    static constexpr int BYTES = OFF_MISC + 16;
    static constexpr int ALLOC = BYTES + 1024;  // room to align the base to 1024
    static_assert(ALLOC <= 227 * 1024, "shared memory");
};

struct FwdParams {
    void *o;
    float *lse;
    unsigned int *status;
    const int *cu_seqlens;         // packed layout: sequence b is rows cu[b] .. cu[b+1]-1
    int varlen, total;             // packed layout flag, rows of all sequences
    int Hq, Hkv, N, nblk, causal;  // N: rows per sequence (packed: the maximum); nblk: 256-row blocks
    int group, planes;             // CTA order (grid_order.cuh): planes per group, B * Hq
    int window;                    // > 0: row r sees keys r - window + 1 .. r only
    int o_f32;                     // O is written in fp32 (before any rounding to the 16-bit type)
    float scale_log2;              // scale * log2(e)
};

constexpr uint32_t kColS = 0, kColO = 256;  // + 128 per tile

// GENERAL = false compiles the sliding window and the packed layout out:
// the dense, full-causal path keeps the leanest issue and softmax loops.
template <int D, bool BF16, bool GENERAL>
__global__ void __launch_bounds__(kThreads, 1)
    fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
               const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
               const FwdParams p) {
    using L = FwdLayout<D>;
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
    const int win = GENERAL ? p.window : 0;
    const bool packed = GENERAL && p.varlen;
    const bool o_f32 = GENERAL && p.o_f32;
    const bool rows_out = packed || o_f32;  // each thread stores its own output row

    // CTA order: planes in L2-sized groups, longest causal blocks first
    int bh, t_lin;
    grid_decode(blockIdx.x, p.planes, p.nblk, p.group, bh, t_lin);
    const int t = p.causal ? (p.nblk - 1 - t_lin) : t_lin;
    const int b = bh / p.Hq;
    const int h = bh - b * p.Hq;
    const int hk = h / (p.Hq / p.Hkv);
    const int q0a = t * 2 * kBM;
    // rows of this sequence: N of them; packed sequences start at row0 of the
    // token-major tensors ("variable length sequence" of the FA3 summary)
    int N = p.N, row0 = 0;
    if (packed) {
        row0 = p.cu_seqlens[b];
        N = p.cu_seqlens[b + 1] - row0;
        if (N < 0 || N > p.N || row0 < 0 || row0 + N > p.total) {
            if (threadIdx.x == 0 && t_lin == 0) record_bad_args(p.status);
            return;  // uniform across the CTA, nothing started yet
        }
    }
    if (q0a >= N) return;  // block past the end of a shorter sequence
    const int nkv_all = (N + kBN - 1) / kBN;
    // K/V tiles each Q tile visits; 0 for a tile that lies entirely past N
    const int nA = p.causal ? min(q0a / kBN + 1, nkv_all) : nkv_all;
    const int nB = q0a + kBM >= N ? 0 : (p.causal ? min((q0a + kBM) / kBN + 1, nkv_all) : nkv_all);
    const int nmax = max(nA, nB);
    // first K/V tile each Q tile visits: with a sliding window of W keys, row
    // r sees keys r - W + 1 .. r, so tile X starts at the tile holding key
    // q0_X - W + 1 (the tiles before it are skipped like those above the
    // causal diagonal)
    const int jA0 = win > 0 ? max(0, q0a - win + 1) / kBN : 0;
    const int jB0 = win > 0 ? max(0, q0a + kBM - win + 1) / kBN : 0;
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
                for (int bx = 0; bx < L::NBOX; ++bx)
                    tma_load_3d(smem + L::OFF_Q + x * L::TILE + bx * L::BOX, &tm_q, q_full, bx * 64,
                                packed ? h : q0a + x * kBM, packed ? row0 + q0a + x * kBM : q_plane);
            // K_j then V_j: the order in which the MMAs first need them
            int nk = 0, nv = 0;
            for (int j = jA0; j < nmax; ++j) {
                const int u = j - jA0;  // position in the K/V stream
                const int ks = u % L::KS;
                if (u >= L::KS && !mbar_wait(&k_empty[ks], ((u / L::KS) + 1) & 1, abort_flag, p.status, 1)) break;
                mbar_arrive_expect_tx(&k_full[ks], L::TILE);
                for (int bx = 0; bx < L::NBOX; ++bx)
                    tma_load_3d(smem + L::OFF_K + ks * L::TILE + bx * L::BOX, &tm_k, &k_full[ks], bx * 64,
                                packed ? hk : j * kBN, packed ? row0 + j * kBN : kv_plane);
                ++nk;
                const int vs = u % L::VS;
                if (u >= L::VS && !mbar_wait(&v_empty[vs], ((u / L::VS) + 1) & 1, abort_flag, p.status, 2)) break;
                mbar_arrive_expect_tx(&v_full[vs], L::TILE);
                for (int bx = 0; bx < L::NBOX; ++bx)
                    tma_load_3d(smem + L::OFF_V + vs * L::TILE + bx * L::BOX, &tm_v, &v_full[vs], bx * 64,
                                packed ? hk : j * kBN, packed ? row0 + j * kBN : kv_plane);
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
            constexpr uint32_t fmt = BF16 ? 1u : 0u;
            constexpr uint32_t idesc_s = make_idesc(kBM, kBN, fmt, false, false);  // K-major both
            constexpr uint32_t idesc_pv = make_idesc(kBM, D, fmt, false, true);    // A tmem, B MN-major
            // one descriptor per operand tile; steps are derived by sdesc_advance
            const uint64_t q_desc0 = make_sdesc_sw128(smem_u32(smem + L::OFF_Q), 16, 1024);
            const uint64_t k_desc0 = make_sdesc_sw128(smem_u32(smem + L::OFF_K), 16, 1024);
            const uint64_t v_desc0 = make_sdesc_sw128(smem_u32(smem + L::OFF_V), L::BOX, 1024);
            int k_ready = -1;  // highest K/V stream position whose K arrival has been observed

            // u = j - jA0 is the position of K/V tile j in the stream
            auto wait_k = [&](int u) -> bool {
                if (u <= k_ready) return true;
                if (!mbar_wait(&k_full[u % L::KS], (u / L::KS) & 1, abort_flag, p.status, 3)) return false;
                tc_fence_after();
                k_ready = u;
                return true;
            };
            // S_x(j) = Q_x K_j^T (A = Q, B = K, both K-major, 32 bytes per step
            // inside a 128-byte row)
            auto issue_s = [&](int x, int u) {
                const uint64_t q_desc = sdesc_advance(q_desc0, x * L::TILE);
                const uint64_t k_desc = sdesc_advance(k_desc0, (u % L::KS) * L::TILE);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t off = (kk >> 2) * L::BOX + (kk & 3) * 32;
                    mma_f16_ss(tmem + kColS + x * 128, sdesc_advance(q_desc, off), sdesc_advance(k_desc, off), idesc_s,
                               kk > 0 ? 1u : 0u);
                }
                mma_commit(&s_full[x]);
            };
            // O_x += P_x V_j (A = P from tensor memory, 16 keys = 8 columns
            // per step; B = V, MN-major, 16 rows of 128 bytes per step); jj is
            // the tile's own step count, u the stream position of V_j
            auto issue_pv = [&](int x, int jj, int u) -> bool {
                if (!mbar_wait(&p_full[x], jj & 1, abort_flag, p.status, 4)) return false;
                tc_fence_after();
                const uint64_t v_desc = sdesc_advance(v_desc0, (u % L::VS) * L::TILE);
                const uint32_t p_col = tmem + kColS + x * 128;
#pragma unroll
                for (int kk = 0; kk < kBN / 16; ++kk)
                    mma_f16_ts(tmem + kColO + x * 128, p_col + kk * 8, sdesc_advance(v_desc, kk * 2048), idesc_pv,
                               (jj > 0 || kk > 0) ? 1u : 0u);
                return true;
            };

            bool ok = mbar_wait(q_full, 0, abort_flag, p.status, 5);
            if (ok) ok = wait_k(0);
            if (ok) {
                issue_s(0, 0);
                if (nB > 0 && jB0 == jA0) issue_s(1, 0);
                mma_commit(&k_empty[0]);
            }
            if (!GENERAL || win == 0) {
                // no window (dense or packed): both tiles start at K/V tile 0
                if (ok && nmax > 0) {
                    ok = mbar_wait(&v_full[0], 0, abort_flag, p.status, 6);
                    tc_fence_after();
                }
                // K_j's slot is released after the first P.V of tile j (one
                // step later than its last reader, S_B(j), needs), and V_{j+1}
                // is checked before S_B(j+1): the issuing thread then goes from
                // the last S MMA of one step straight to the first P.V of the next
                for (int j = 0; ok && j < nmax; ++j) {
                    // V_j is ready here
                    if (j < nA) {
                        if (!issue_pv(0, j, j)) { ok = false; break; }
                    }
                    if (j >= 1) mma_commit(&k_empty[j % L::KS]);  // K_j: last read by S_B(j)
                    if (j + 1 < nA) {
                        if (!wait_k(j + 1)) { ok = false; break; }
                        issue_s(0, j + 1);
                    } else if (j < nA) {
                        mma_commit(&o_final[0]);
                    }
                    if (j < nB) {
                        if (!issue_pv(1, j, j)) { ok = false; break; }
                    }
                    mma_commit(&v_empty[j % L::VS]);
                    if (j + 1 < nmax) {
                        if (!mbar_wait(&v_full[(j + 1) % L::VS], ((j + 1) / L::VS) & 1, abort_flag, p.status, 6)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                    }
                    if (j + 1 < nB) {
                        if (!wait_k(j + 1)) { ok = false; break; }
                        issue_s(1, j + 1);
                    } else if (j < nB) {
                        mma_commit(&o_final[1]);
                    }
                }
            } else {
                for (int j = jA0; ok && j < nmax; ++j) {
                    const int u = j - jA0;
                    if (!mbar_wait(&v_full[u % L::VS], (u / L::VS) & 1, abort_flag, p.status, 6)) { ok = false; break; }
                    tc_fence_after();
                    for (int x = 0; x < 2; ++x) {
                        const int nx = x ? nB : nA;
                        const int jx0 = x ? jB0 : jA0;
                        if (j < jx0 - 1 || j >= nx) continue;
                        if (j >= jx0) {
                            if (!issue_pv(x, j - jx0, u)) { ok = false; break; }
                            if (j + 1 == nx) mma_commit(&o_final[x]);
                        }
                        if (j + 1 < nx) {
                            // S_x(j+1) overwrites P_x(j), which the MMAs just issued read first
                            if (!wait_k(u + 1)) { ok = false; break; }
                            issue_s(x, u + 1);
                        }
                    }
                    if (!ok) break;
                    mma_commit(&v_empty[u % L::VS]);
                    if (j + 1 < nmax) mma_commit(&k_empty[(u + 1) % L::KS]);
                }
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
        const int jx0 = x ? jB0 : jA0;
        const float sl2 = p.scale_log2;
        float m_ref = -INFINITY;
        float l_sum = 0.0f;    // sum of the rounded P fed to the MMA: normalises O
        float l_exact = 0.0f;  // sum of the unrounded P: gives L
        bool ok = true;

        for (int j = jx0; ok && j < nx; ++j) {
            const int jj = j - jx0;  // this tile's own step count
            // every lane waits, then the warp votes: the tcgen05.ld/st below
            // are warp-collective (.sync.aligned) and need all 32 lanes
            const bool got_s = mbar_wait(&s_full[x], jj & 1, abort_flag, p.status, 7);
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
            const bool need_mask = (kv0 + kBN > N) || (p.causal && kv0 + kBN - 1 > q0) ||
                                   (win > 0 && kv0 < q0 + kBM - win);
            if (need_mask) {
                // visible: lo <= key < hi
                const int hi = p.causal ? min(N, q0 + row + 1) : N;
                const int lo = win > 0 ? q0 + row - win + 1 : 0;
#pragma unroll
                for (int c = 0; c < 128; ++c)
                    if (kv0 + c >= hi || kv0 + c < lo) s[c] = __float_as_uint(-INFINITY);
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
            __syncwarp();  // reconverge after the per-row branches above
            // a row that has seen no visible key yet (its keys start in a later
            // tile of a sliding window) keeps m_ref = -inf: use 0 so that its
            // masked scores give P = 0 rather than -inf - (-inf)
            const float m_use = (GENERAL && m_ref == -INFINITY) ? 0.0f : m_ref;
            const float2 neg_m = make_float2(-m_use, -m_use);
            const float2 sl2x2 = make_float2(sl2, sl2);
            float2 lr01 = make_float2(0.f, 0.f), lr23 = lr01, le01 = lr01, le23 = lr01;
            // P is written back in chunks of CH scores (CH / 2 packed columns),
            // which keeps fewer registers live than one 64-column store
            constexpr int CH = 32;
#pragma unroll
            for (int hh = 0; hh < 128 / CH; ++hh) {
                uint32_t pk[CH / 2];
#pragma unroll
                for (int c = CH * hh; c < CH * hh + CH; c += 4) {
                    const float2 x01 =
                        ffma2(make_float2(__uint_as_float(s[c]), __uint_as_float(s[c + 1])), sl2x2, neg_m);
                    const float2 x23 =
                        ffma2(make_float2(__uint_as_float(s[c + 2]), __uint_as_float(s[c + 3])), sl2x2, neg_m);
                    const float p0 = ex2_approx(x01.x);
                    const float p1 = ex2_approx(x01.y);
                    const float p2 = ex2_approx(x23.x);
                    const float p3 = ex2_approx(x23.y);
                    const int k = (c - CH * hh) / 2;
                    // l sums the rounded P that the MMA consumes, so O~ / l is an
                    // exactly normalised mix of V rows even when one term dominates
                    if constexpr (BF16) {
                        pk[k] = pack_bf16x2(p0, p1);
                        pk[k + 1] = pack_bf16x2(p2, p3);
                    } else {
                        pk[k] = pack_f16x2(p0, p1);
                        pk[k + 1] = pack_f16x2(p2, p3);
                    }
                    if constexpr (BF16) {
                        lr01 = add_bf16x2_f32x2(pk[k], lr01);
                        lr23 = add_bf16x2_f32x2(pk[k + 1], lr23);
                    } else {
                        lr01 = fadd2(lr01, unpack2<BF16>(pk[k]));
                        lr23 = fadd2(lr23, unpack2<BF16>(pk[k + 1]));
                    }
                    le01 = fadd2(le01, make_float2(p0, p1));
                    le23 = fadd2(le23, make_float2(p2, p3));
                }
                // P of keys CH hh .. + CH - 1 -> columns CH / 2 * hh .. of this
                // row's S, all of which have been read
                if constexpr (CH == 64)
                    tmem_st_x32(lane_base + col_s + 32 * hh, pk);
                else
                    tmem_st_x16(lane_base + col_s + 16 * hh, pk);
            }
            l_sum += (lr01.x + lr01.y) + (lr23.x + lr23.y);
            l_exact += (le01.x + le01.y) + (le23.x + le23.y);
            // O_x already holds P_x(0..j-1) V (S_x(j) was issued after the last
            // P.V of this tile), and P_x(j) V is issued only after p_full;
            // warp-uniform branch, lanes that keep their max use alpha = 1
            if (jj >= 1 && __any_sync(0xffffffffu, rescale)) {
                // one tensor-memory round trip: the S registers are free again
                uint32_t o[D];
#pragma unroll
                for (int c0 = 0; c0 < D; c0 += 32) tmem_ld_x32(lane_base + col_o + c0, o + c0);
#pragma unroll
                for (int c0 = 0; c0 < D; c0 += 32) tmem_ld_wait_x32(o + c0);
#pragma unroll
                for (int c = 0; c < D; c += 2) {
                    const float2 r = fmul2(make_float2(__uint_as_float(o[c]), __uint_as_float(o[c + 1])),
                                           make_float2(alpha, alpha));
                    o[c] = __float_as_uint(r.x);
                    o[c + 1] = __float_as_uint(r.y);
                }
#pragma unroll
                for (int c0 = 0; c0 < D; c0 += 32) tmem_st_x32(lane_base + col_o + c0, o + c0);
            }
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(&p_full[x]);
        }

        if (nx > 0) {  // uniform across the warpgroup
            if (ok) ok = mbar_wait(&o_final[x], 0, abort_flag, p.status, 9);
            __syncwarp();
            // uniform decision across the tile's 128 threads (the epilogue has a
            // named barrier that all of them must reach)
            ok = named_bar_and(1 + x, kBM, ok);
            if (ok) {
                tc_fence_after();
                // Epilogue: O = O~ / l, staged through the (now idle) Q buffer of
                // this tile in the 128-byte-swizzled layout of the output TMA box.
                const float inv_l = 1.0f / l_sum;
                uint8_t *stage = smem + L::OFF_Q + x * L::TILE;
#pragma unroll 1
                for (int c0 = 0; c0 < D; c0 += 32) {
                    uint32_t o[32];
                    tmem_ld_x32(lane_base + col_o + c0, o);
                    tmem_ld_wait_x32(o);
#pragma unroll
                    for (int c = 0; c < 32; ++c) o[c] = __float_as_uint(__uint_as_float(o[c]) * inv_l);
                    uint32_t w[16];
#pragma unroll
                    for (int c = 0; c < 16; ++c)
                        w[c] = BF16 ? pack_bf16x2(__uint_as_float(o[2 * c]), __uint_as_float(o[2 * c + 1]))
                                    : pack_f16x2(__uint_as_float(o[2 * c]), __uint_as_float(o[2 * c + 1]));
                    if (rows_out) {
                        // packed rows: a 128-row box past this sequence's end
                        // would overwrite the next sequence; fp32 rows: the box
                        // is laid out for 16-bit elements.  So each thread
                        // stores its own row (16-byte stores).
                        if (q0 + row < N) {
                            const size_t r = packed ? (size_t)(row0 + q0 + row) * p.Hq + h
                                                    : (size_t)q_plane * N + q0 + row;
                            if (o_f32) {
                                uint4 *dst = reinterpret_cast<uint4 *>(static_cast<float *>(p.o) + r * D + c0);
#pragma unroll
                                for (int q = 0; q < 8; ++q)
                                    dst[q] = make_uint4(o[4 * q], o[4 * q + 1], o[4 * q + 2], o[4 * q + 3]);
                            } else {
                                uint4 *dst =
                                    reinterpret_cast<uint4 *>(static_cast<uint8_t *>(p.o) + r * (D * 2)) + c0 / 8;
#pragma unroll
                                for (int q = 0; q < 4; ++q)
                                    dst[q] = make_uint4(w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]);
                            }
                        }
                    } else {
                        uint8_t *rowp = stage + (c0 >> 6) * L::BOX + row * 128;
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            const int chunk = ((c0 & 63) >> 3) + q;
                            *reinterpret_cast<uint4 *>(rowp + ((chunk ^ (row & 7)) << 4)) =
                                make_uint4(w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]);
                        }
                    }
                }
                if (!rows_out) {
                    fence_proxy_async_smem();
                    named_bar_sync(1 + x, kBM);
                    if (row == 0) {
                        for (int bx = 0; bx < L::NBOX; ++bx)
                            tma_store_3d(&tm_o, stage + bx * L::BOX, bx * 64, q0, q_plane);
                        bulk_commit();
                        bulk_wait_read_all();
                    }
                }
                if (q0 + row < N) {
                    const size_t li = packed ? (size_t)h * p.total + row0 + q0 + row : (size_t)q_plane * N + q0 + row;
                    p.lse[li] = (m_ref + log2f(l_exact)) * 0.69314718055994530942f;
                }
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

template <int D, bool BF16>
cudaError_t launch_fwd_t(const FwdArgs &a, cudaStream_t st) {
    using L = FwdLayout<D>;
    const CUtensorMapDataType dt = BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    CUtensorMap tq, tk, tv, to;
    if (!make_tmap_tiles(&tq, a.q, dt, D, a.lay, a.Hq, kBM) || !make_tmap_tiles(&tk, a.k, dt, D, a.lay, a.Hkv, kBN) ||
        !make_tmap_tiles(&tv, a.v, dt, D, a.lay, a.Hkv, kBN) || !make_tmap_tiles(&to, a.o, dt, D, a.lay, a.Hq, kBM))
        return cudaErrorInvalidValue;
    const bool general = a.window > 0 || a.lay.varlen || a.o_f32;
    auto kernel = general ? fwd_kernel<D, BF16, true> : fwd_kernel<D, BF16, false>;
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, L::ALLOC);
    if (e != cudaSuccess) return e;
    FwdParams p;
    p.o = a.o;
    p.lse = a.lse;
    p.status = device_status_ptr();
    p.cu_seqlens = a.lay.cu_seqlens;
    p.varlen = a.lay.varlen;
    p.total = a.lay.total;
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
    p.window = a.window;
    p.o_f32 = a.o_f32 ? 1 : 0;
    p.scale_log2 = a.scale * 1.4426950408889634f;
    const long long grid = (long long)p.nblk * a.B * a.Hq;
    kernel<<<dim3((unsigned)grid), dim3(kThreads), L::ALLOC, st>>>(tq, tk, tv, to, p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd(const FwdArgs &a, cudaStream_t st) {
    // Short sequences go to the persistent kernel (fa_fwd_persist.cu, same
    // results bit for bit): with few K/V tiles per 256-row block, the set-up
    // and epilogue it overlaps across blocks weigh most.  Crossover measured
    // on a GB300 (bf16, d = 128, 16 heads, L2 flushed): causal N = 512 / 1024
    // / 2048 ran 1.3x / 1.1x / 1.01-1.03x faster than one CTA per block,
    // N = 3072 / 4096 / 8192 0.99x / 0.98x / 0.97x; without the mask
    // N = 1024 1.08x, N = 2048 1.02x, N = 4096 0.97x.
    // The same holds for a sliding window (a block walks at most about
    // W / 128 + 2 K/V tiles whatever N is) and for packed batches: at
    // N = 8192, W = 256 / 1024 / 4096 ran 1.10x / 1.05x / 0.96x; a packed
    // batch of lengths up to 2048 1.01x, up to 7506 0.96x.
    // It stores O rows in 32-byte pieces, so it needs O 32-byte aligned (the
    // entry points promise only 16).
    const bool o32 = (reinterpret_cast<uintptr_t>(a.o) & 31u) == 0;
    const int walk = a.window > 0 ? (a.window < a.N ? a.window : a.N) : a.N;  // keys a block's rows see
    if (!a.o_f32 && o32 && walk <= 2048) return launch_fwd_persist(a, st);
    if (a.d == 128) return a.bf16 ? launch_fwd_t<128, true>(a, st) : launch_fwd_t<128, false>(a, st);
    if (a.d == 64) return a.bf16 ? launch_fwd_t<64, true>(a, st) : launch_fwd_t<64, false>(a, st);
    return cudaErrorInvalidValue;
}

}  // namespace fa
