// fa_fwd_persist.cu -- persistent FlashAttention-2 forward for sm_103a with a
// dynamic, longest-first block schedule (dense or packed layout, causal, full
// or causal sliding-window mask, bf16 / fp16, d = 64 or 128, 16-bit output).
//
// The FlashAttention-3 summary page ("remaining optimisations": persistent
// kernel) names a persistent kernel as the way to keep the tensor cores busy
// across the end of one tile and the start of the next.  The plain forward
// (fa_fwd.cu) starts one CTA per 256-row block: every CTA pays its set-up
// (barriers, tensor memory, the first Q and K/V loads) and its epilogue with
// nothing overlapping them, which costs most on short sequences, where a
// block walks few K/V tiles.
//
// Here the grid still has one CTA per block, in the same longest-first,
// L2-grouped order (grid_order.cuh), but every CTA that runs keeps running:
// while it works on a block it asks the hardware (cluster launch control,
// clusterlaunchcontrol.try_cancel) to cancel a CTA that has not been launched
// yet and takes that CTA's block next.  The blocks are therefore handed out
// dynamically in launch order -- the longest causal blocks first -- with no
// counter in global memory.  Across blocks the K/V ring, the barrier phases
// and the tensor-memory allocation carry on: Q_x of the next block is loaded
// as soon as the last S_x MMA of the current one has completed, the next
// block's S_A(0) and S_B(0) are issued right after the current block's last
// P.V MMAs, and each softmax warpgroup's epilogue (O = O~ / l, L = m + ln l)
// runs while the tensor cores work on the other tile and on the next block.
// O rows are stored by their own threads, one whole 32-byte sector per store
// (the Q buffer that stages O in the plain forward is already being
// refilled).
//
// Per block the arithmetic is that of fa_fwd.cu (two 128-row Q tiles A and B
// walking the same K/V stream, ping-ponged softmax warpgroups, exact lazy
// rescale by more than 8 in log2 units, P in 16 bits from tensor memory): the
// outputs are bit-identical to the plain forward's.
// GENERAL instances add the causal sliding window (a block's K/V stream starts
// at the tile holding its first row's oldest visible key) and packed
// variable-length batches (token-major rows from cu_seqlens; blocks past a
// sequence's end are empty items, taken and dropped like any other), the two
// cases of the FlashAttention-3 summary's GQA / sliding-window and
// variable-length discussions whose blocks walk few K/V tiles whatever N is.
// Warps: 0-3 softmax + epilogue of tile A, 4-7 of tile B, 8 TMA producer and
// scheduler, 9 MMA issuer (owns the tensor memory).
#include "grid_order.cuh"
#include "host_util.h"
#include "ptx.cuh"

namespace fa {

namespace {

constexpr int kBM = 128;       // query rows per Q tile (TMEM lanes)
constexpr int kBN = 128;       // keys per K/V tile
constexpr int kThreads = 320;  // 10 warps
constexpr int kProducerWarp = 8, kMmaWarp = 9;
constexpr int kSoftmaxWarps = 8;
constexpr float kRescaleThreshold = 8.0f;

template <int D>
struct PersistLayout {
    static constexpr int KS = D == 128 ? 3 : 4;  // K ring depth
    static constexpr int VS = D == 128 ? 2 : 4;  // V ring depth
    static constexpr int NBOX = D / 64;
    static constexpr int TILE = 128 * D * 2;
    static constexpr int BOX = 128 * 128;
    static constexpr int OFF_Q = 0;  // Q_A, then Q_B
    static constexpr int OFF_K = OFF_Q + 2 * TILE;
    static constexpr int OFF_V = OFF_K + KS * TILE;
    static constexpr int OFF_BAR = OFF_V + VS * TILE;
    // q_full[2], q_empty[2], k_full[KS], k_empty[KS], v_full[VS], v_empty[VS],
    // s_full[2], p_full[2], o_final[2], item_full[2], item_empty[2], clc, drain
    static constexpr int NBAR = 2 + 2 + 2 * KS + 2 * VS + 2 + 2 + 2 + 2 + 2 + 1 + 1;
    static constexpr int OFF_CLC = OFF_BAR + NBAR * 8;   // 16-byte cancellation response
    // item slots [2] of {item, first row, rows} (16 bytes each), TMEM base, abort flag
    static constexpr int OFF_MISC = OFF_CLC + 16;
    static constexpr int BYTES = OFF_MISC + 48;
    static constexpr int ALLOC = BYTES + 1024;  // room to align the base to 1024
    static_assert(OFF_CLC % 16 == 0, "response alignment");
    static_assert(ALLOC <= 227 * 1024, "shared memory");
};

struct PersistParams {
    void *o;
    float *lse;
    unsigned int *status;
    const int *cu_seqlens;  // packed batches: [B + 1] row offsets
    int varlen, total;      // packed layout; its total rows
    int window;             // 0: none, else a causal window of that many keys
    int Hq, Hkv, N, nblk, causal;  // N: rows per sequence (packed: the maximum)
    int group, planes;             // CTA order (grid_order.cuh)
    float scale_log2;
};

constexpr uint32_t kColS = 0, kColO = 256;  // + 128 per tile

// Cluster launch control: ask for the cancellation of a CTA that has not been
// launched yet; the 16-byte response lands in shared memory and completes
// `bar` (16 transaction bytes).
__device__ __forceinline__ void clc_try_cancel(void *resp, uint64_t *bar) {
    asm volatile(
        "clusterlaunchcontrol.try_cancel.async.shared::cta.mbarrier::complete_tx::bytes.b128 [%0], [%1];" ::"r"(
            smem_u32(resp)),
        "r"(smem_u32(bar))
        : "memory");
}

// Reads a completed response: the canceled CTA's x index, or -1 if nothing
// was left to cancel.
__device__ __forceinline__ int clc_result(const void *resp) {
    uint32_t canceled, x;
    asm volatile(
        "{\n\t.reg .pred p;\n\t.reg .b128 r;\n\t"
        "ld.shared.b128 r, [%2];\n\t"
        "clusterlaunchcontrol.query_cancel.is_canceled.pred.b128 p, r;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t"
        "mov.u32 %1, 0;\n\t"
        "@p clusterlaunchcontrol.query_cancel.get_first_ctaid.v4.b32.b128 {%1, _, _, _}, r;\n\t}\n"
        : "=r"(canceled), "=r"(x)
        : "r"(smem_u32(resp))
        : "memory");
    return canceled ? (int)x : -1;
}

// The block an item index stands for (the plain forward's grid order), in a
// sequence of n rows starting at token row0 (dense: row0 = 0, n = N).  Tile x
// walks K/V tiles jx0 .. nx - 1 (none if nx = 0); the block's K/V stream is
// tiles jA0 .. nmax - 1 (jB0 >= jA0, nB >= nA whenever tile B has work).
struct Block {
    int bh, q0a, jA0, jB0, nA, nB, nmax, row0, n;
};

__device__ __forceinline__ Block decode_block(int item, int row0, int n, const PersistParams &p) {
    Block blk;
    int t_lin;
    grid_decode(item, p.planes, p.nblk, p.group, blk.bh, t_lin);
    const int t = p.causal ? (p.nblk - 1 - t_lin) : t_lin;
    blk.q0a = t * 2 * kBM;
    blk.row0 = row0;
    blk.n = n;
    blk.jA0 = blk.jB0 = 0;
    if (blk.q0a >= n) {  // past the end of a shorter packed sequence: no work
        blk.nA = blk.nB = blk.nmax = 0;
        return blk;
    }
    const int nkv_all = (n + kBN - 1) / kBN;
    blk.nA = p.causal ? min(blk.q0a / kBN + 1, nkv_all) : nkv_all;
    blk.nB = blk.q0a + kBM >= n ? 0 : (p.causal ? min((blk.q0a + kBM) / kBN + 1, nkv_all) : nkv_all);
    blk.nmax = max(blk.nA, blk.nB);
    if (p.window > 0) {
        // row r sees keys r - W + 1 .. r: tile x starts at the tile holding
        // key q0_x - W + 1 (the tiles before it are skipped like those above
        // the causal diagonal)
        blk.jA0 = max(0, blk.q0a - p.window + 1) / kBN;
        blk.jB0 = max(0, blk.q0a + kBM - p.window + 1) / kBN;
    }
    return blk;
}

template <int D, bool BF16, bool GENERAL>
__global__ void __launch_bounds__(kThreads, 1)
    fwd_persist_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v, const PersistParams p) {
    using L = PersistLayout<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::OFF_BAR);
    uint64_t *q_full = bars;          // [2]
    uint64_t *q_empty = q_full + 2;   // [2]
    uint64_t *k_full = q_empty + 2;
    uint64_t *k_empty = k_full + L::KS;
    uint64_t *v_full = k_empty + L::KS;
    uint64_t *v_empty = v_full + L::VS;
    uint64_t *s_full = v_empty + L::VS;  // [2]
    uint64_t *p_full = s_full + 2;       // [2]
    uint64_t *o_final = p_full + 2;      // [2]
    uint64_t *item_full = o_final + 2;   // [2]
    uint64_t *item_empty = item_full + 2;  // [2]
    uint64_t *clc_bar = item_empty + 2;
    uint64_t *drain = clc_bar + 1;
    void *clc_resp = smem + L::OFF_CLC;
    volatile int *item_slot = reinterpret_cast<volatile int *>(smem + L::OFF_MISC);  // [2][4]
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L::OFF_MISC + 32);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::OFF_MISC + 36);
    const bool packed = GENERAL && p.varlen;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int x = 0; x < 2; ++x) {
            mbar_init(&q_full[x], 1);
            mbar_init(&q_empty[x], 1);
            mbar_init(&s_full[x], 1);
            mbar_init(&p_full[x], kBM);
            mbar_init(&o_final[x], 1);
            mbar_init(&item_full[x], 1);
            mbar_init(&item_empty[x], 1 + kSoftmaxWarps);  // the MMA thread + lane 0 of each softmax warp
        }
        for (int s = 0; s < L::KS; ++s) { mbar_init(&k_full[s], 1); mbar_init(&k_empty[s], 1); }
        for (int s = 0; s < L::VS; ++s) { mbar_init(&v_full[s], 1); mbar_init(&v_empty[s], 1); }
        mbar_init(clc_bar, 1);
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
        // ---------------------------------------- TMA producer and scheduler
        if (lane == 0) {
            prefetch_tmap(&tm_q);
            prefetch_tmap(&tm_k);
            prefetch_tmap(&tm_v);
            int item = blockIdx.x;  // this CTA's own block first
            int nq[2] = {0, 0};     // blocks so far that had tile x (q_full / q_empty phases)
            int u_base = 0;         // K/V stream position of the block's first tile
            int nk = 0, nv = 0;     // K / V copies issued
            int clc_n = 0;          // cancellation requests whose response was read
            bool clc_pending = false;
            bool ok = true;
            for (int k = 0; ok; ++k) {
                // publish the block to the other roles (two slots)
                const int slot = k & 1;
                if (k >= 2 && !mbar_wait(&item_empty[slot], ((k >> 1) - 1) & 1, abort_flag, p.status, 60)) break;
                // the block's sequence: packed batches read its bounds once, here
                int row0 = 0, n = p.N;
                if (packed && item >= 0) {
                    int plane, t_lin;
                    grid_decode(item, p.planes, p.nblk, p.group, plane, t_lin);
                    const int b = plane / p.Hq;
                    row0 = p.cu_seqlens[b];
                    n = p.cu_seqlens[b + 1] - row0;
                    if (n < 0 || n > p.N || row0 < 0 || row0 + n > p.total) {
                        record_bad_args(p.status);
                        row0 = 0;
                        n = 0;  // no work for this block
                    }
                }
                item_slot[4 * slot] = item;
                item_slot[4 * slot + 1] = row0;
                item_slot[4 * slot + 2] = n;
                mbar_arrive(&item_full[slot]);  // release: the slot writes are seen by every waiter
                if (item < 0) break;
                // ask for the next block while this one's tiles load
                mbar_arrive_expect_tx(clc_bar, 16);
                clc_try_cancel(clc_resp, clc_bar);
                clc_pending = true;
                const Block blk = decode_block(item, row0, n, p);
                const int b = blk.bh / p.Hq;
                const int h = blk.bh - b * p.Hq;
                const int hk = h / (p.Hq / p.Hkv);
                const int kv_plane = b * p.Hkv + hk;
                // Q_x: its buffer is free once the previous block's last S_x MMA has completed
                for (int x = 0; x < 2 && ok; ++x) {
                    if ((x ? blk.nB : blk.nA) == 0) continue;
                    if (nq[x] > 0 && !mbar_wait(&q_empty[x], (nq[x] - 1) & 1, abort_flag, p.status, 61)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&q_full[x], L::TILE);
                    const int qr = blk.q0a + x * kBM;
                    for (int bx = 0; bx < L::NBOX; ++bx)
                        tma_load_3d(smem + L::OFF_Q + x * L::TILE + bx * L::BOX, &tm_q, &q_full[x], bx * 64,
                                    packed ? h : qr, packed ? row0 + qr : blk.bh);
                    ++nq[x];
                }
                // K_j then V_j, continuing the ring positions of earlier blocks
                for (int j = blk.jA0; ok && j < blk.nmax; ++j) {
                    const int u = u_base + (j - blk.jA0);
                    const int ks = u % L::KS;
                    if (u >= L::KS && !mbar_wait(&k_empty[ks], ((u / L::KS) + 1) & 1, abort_flag, p.status, 62)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&k_full[ks], L::TILE);
                    for (int bx = 0; bx < L::NBOX; ++bx)
                        tma_load_3d(smem + L::OFF_K + ks * L::TILE + bx * L::BOX, &tm_k, &k_full[ks], bx * 64,
                                    packed ? hk : j * kBN, packed ? row0 + j * kBN : kv_plane);
                    ++nk;
                    const int vs = u % L::VS;
                    if (u >= L::VS && !mbar_wait(&v_empty[vs], ((u / L::VS) + 1) & 1, abort_flag, p.status, 63)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&v_full[vs], L::TILE);
                    for (int bx = 0; bx < L::NBOX; ++bx)
                        tma_load_3d(smem + L::OFF_V + vs * L::TILE + bx * L::BOX, &tm_v, &v_full[vs], bx * 64,
                                    packed ? hk : j * kBN, packed ? row0 + j * kBN : kv_plane);
                    ++nv;
                }
                if (!ok) break;
                u_base += blk.nmax - blk.jA0;
                // the next block: the one whose CTA was canceled, or none
                if (!mbar_wait(clc_bar, clc_n & 1, abort_flag, p.status, 64)) break;
                ++clc_n;
                clc_pending = false;
                item = clc_result(clc_resp);
            }
            if (*abort_flag) {
                // let copies and the cancellation request in flight land first
                for (int x = 0; x < 2; ++x)
                    if (nq[x] > 0) mbar_wait_drain(&q_full[x], (nq[x] - 1) & 1, 10000000ull);
                for (int u = max(0, nk - L::KS); u < nk; ++u)
                    mbar_wait_drain(&k_full[u % L::KS], (u / L::KS) & 1, 10000000ull);
                for (int u = max(0, nv - L::VS); u < nv; ++u)
                    mbar_wait_drain(&v_full[u % L::VS], (u / L::VS) & 1, 10000000ull);
                if (clc_pending) mbar_wait_drain(clc_bar, clc_n & 1, 10000000ull);
            }
        }
        __syncwarp();
    } else if (warp == kMmaWarp) {
        // ------------------------------------------------------- MMA issuer
        if (lane == 0) {
            constexpr uint32_t fmt = BF16 ? 1u : 0u;
            constexpr uint32_t idesc_s = make_idesc(kBM, kBN, fmt, false, false);  // K-major both
            constexpr uint32_t idesc_pv = make_idesc(kBM, D, fmt, false, true);    // A tmem, B MN-major
            const uint64_t q_desc0 = make_sdesc_sw128(smem_u32(smem + L::OFF_Q), 16, 1024);
            const uint64_t k_desc0 = make_sdesc_sw128(smem_u32(smem + L::OFF_K), 16, 1024);
            const uint64_t v_desc0 = make_sdesc_sw128(smem_u32(smem + L::OFF_V), L::BOX, 1024);
            int k_ready = -1;       // highest K stream position whose arrival has been observed
            int gs[2] = {0, 0};     // S / P steps issued so far per tile (s_full, p_full phases)
            int nq[2] = {0, 0};     // blocks so far that had tile x (q_full phases)
            int u_base = 0;

            auto wait_k = [&](int u) -> bool {
                if (u <= k_ready) return true;
                if (!mbar_wait(&k_full[u % L::KS], (u / L::KS) & 1, abort_flag, p.status, 65)) return false;
                tc_fence_after();
                k_ready = u;
                return true;
            };
            // S_x = Q_x K_u^T into tile x's S columns
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
            // O_x (+)= P_x V_u once the softmax warps have written P_x (global
            // step g of tile x); the block's first step overwrites O_x
            auto issue_pv = [&](int x, bool first, int u) -> bool {
                if (!mbar_wait(&p_full[x], gs[x] & 1, abort_flag, p.status, 66)) return false;
                ++gs[x];
                tc_fence_after();
                const uint64_t v_desc = sdesc_advance(v_desc0, (u % L::VS) * L::TILE);
                const uint32_t p_col = tmem + kColS + x * 128;
#pragma unroll
                for (int kk = 0; kk < kBN / 16; ++kk)
                    mma_f16_ts(tmem + kColO + x * 128, p_col + kk * 8, sdesc_advance(v_desc, kk * 2048), idesc_pv,
                               (!first || kk > 0) ? 1u : 0u);
                return true;
            };
            auto wait_q = [&](int x) -> bool {
                if (!mbar_wait(&q_full[x], nq[x] & 1, abort_flag, p.status, 67)) return false;
                ++nq[x];
                tc_fence_after();
                return true;
            };

            bool ok = true;
            for (int k = 0; ok; ++k) {
                const int slot = k & 1;
                if (!mbar_wait(&item_full[slot], (k >> 1) & 1, abort_flag, p.status, 68)) break;
                const int item = item_slot[4 * slot];
                const int row0 = item_slot[4 * slot + 1], n = item_slot[4 * slot + 2];
                mbar_arrive(&item_empty[slot]);
                if (item < 0) break;
                const Block blk = decode_block(item, row0, n, p);
                const int nA = blk.nA, nB = blk.nB, nmax = blk.nmax;
                if (GENERAL && p.window > 0) {
                    // the plain forward's general schedule: per K/V tile j (stream
                    // position u), for each tile x that has work there,
                    // O_x += P_x V_j, then S_x(j+1); a tile whose window starts one
                    // K/V tile later has its first S issued in the step before
                    if (nmax == 0) continue;  // empty block
                    const int jA0 = blk.jA0, jB0 = blk.jB0;
                    if (!(ok = wait_q(0) && wait_k(u_base))) break;
                    issue_s(0, u_base);
                    if (nA - jA0 == 1) mma_commit(&q_empty[0]);
                    if (nB > 0 && jB0 == jA0) {
                        if (!(ok = wait_q(1))) break;
                        issue_s(1, u_base);
                        if (nB - jB0 == 1) mma_commit(&q_empty[1]);
                    }
                    mma_commit(&k_empty[u_base % L::KS]);
                    for (int j = jA0; ok && j < nmax; ++j) {
                        const int u = u_base + (j - jA0);
                        if (!mbar_wait(&v_full[u % L::VS], (u / L::VS) & 1, abort_flag, p.status, 69)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        for (int x = 0; x < 2; ++x) {
                            const int nx = x ? nB : nA;
                            const int jx0 = x ? jB0 : jA0;
                            if (nx == 0 || j < jx0 - 1 || j >= nx) continue;
                            if (j >= jx0) {
                                if (!issue_pv(x, j == jx0, u)) { ok = false; break; }
                                if (j + 1 == nx) mma_commit(&o_final[x]);
                            }
                            if (j + 1 < nx) {
                                // S_x(j+1) overwrites P_x(j), which the MMAs just issued read first
                                if (j + 1 == jx0 && !wait_q(x)) { ok = false; break; }
                                if (!wait_k(u + 1)) { ok = false; break; }
                                issue_s(x, u + 1);
                                if (j + 2 == nx) mma_commit(&q_empty[x]);
                            }
                        }
                        if (!ok) break;
                        mma_commit(&v_empty[u % L::VS]);
                        if (j + 1 < nmax) mma_commit(&k_empty[(u + 1) % L::KS]);
                    }
                    u_base += nmax - jA0;
                    continue;
                }
                if (nmax == 0) continue;  // a packed block past its sequence's end
                // first S of both tiles (the previous block's last P.V MMAs run first)
                if (nA > 0) {
                    if (!(ok = wait_q(0) && wait_k(u_base))) break;
                    issue_s(0, u_base);
                    if (nA == 1) mma_commit(&q_empty[0]);  // last reader of Q_A in this block
                }
                if (nB > 0) {
                    if (!(ok = wait_q(1) && wait_k(u_base))) break;
                    issue_s(1, u_base);
                    if (nB == 1) mma_commit(&q_empty[1]);
                }
                mma_commit(&k_empty[u_base % L::KS]);
                if (!mbar_wait(&v_full[u_base % L::VS], (u_base / L::VS) & 1, abort_flag, p.status, 69)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                // the plain forward's dense schedule: per K/V tile j, O_A += P_A V_j,
                // S_A(j+1), O_B += P_B V_j, S_B(j+1)
                for (int j = 0; ok && j < nmax; ++j) {
                    const int u = u_base + j;
                    if (j < nA && !issue_pv(0, j == 0, u)) { ok = false; break; }
                    if (j >= 1) mma_commit(&k_empty[u % L::KS]);  // K_j: last read by S_B(j)
                    if (j + 1 < nA) {
                        if (!wait_k(u + 1)) { ok = false; break; }
                        issue_s(0, u + 1);
                        if (j + 2 == nA) mma_commit(&q_empty[0]);
                    } else if (j < nA) {
                        mma_commit(&o_final[0]);
                    }
                    if (j < nB && !issue_pv(1, j == 0, u)) { ok = false; break; }
                    mma_commit(&v_empty[u % L::VS]);
                    if (j + 1 < nmax) {
                        if (!mbar_wait(&v_full[(u + 1) % L::VS], ((u + 1) / L::VS) & 1, abort_flag, p.status, 69)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                    }
                    if (j + 1 < nB) {
                        if (!wait_k(u + 1)) { ok = false; break; }
                        issue_s(1, u + 1);
                        if (j + 2 == nB) mma_commit(&q_empty[1]);
                    } else if (j < nB) {
                        mma_commit(&o_final[1]);
                    }
                }
                u_base += nmax;
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
        const float sl2 = p.scale_log2;
        int gs = 0;  // this tile's S steps seen so far (s_full phases)
        int nf = 0;  // blocks so far in which this tile had work (o_final phases)
        bool ok = true;
        for (int k = 0; ok; ++k) {
            const int slot = k & 1;
            const bool got = mbar_wait(&item_full[slot], (k >> 1) & 1, abort_flag, p.status, 70);
            if (!__all_sync(0xffffffffu, got)) break;
            const int item = item_slot[4 * slot];
            const int row0 = item_slot[4 * slot + 1], n = item_slot[4 * slot + 2];
            __syncwarp();
            if (lane == 0) mbar_arrive(&item_empty[slot]);
            if (item < 0) break;
            const Block blk = decode_block(item, row0, n, p);
            const int q0 = blk.q0a + x * kBM;
            const int nx = x ? blk.nB : blk.nA;
            const int jx0 = GENERAL ? (x ? blk.jB0 : blk.jA0) : 0;
            if (nx == 0) continue;
            const int win = GENERAL ? p.window : 0;
            float m_ref = -INFINITY;
            float l_sum = 0.0f;    // sum of the rounded P fed to the MMA: normalises O
            float l_exact = 0.0f;  // sum of the unrounded P: gives L
            for (int j = jx0; j < nx; ++j) {
                const bool got_s = mbar_wait(&s_full[x], gs & 1, abort_flag, p.status, 71);
                if (!__all_sync(0xffffffffu, got_s)) { ok = false; break; }
                ++gs;
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
                if ((kv0 + kBN > n) || (p.causal && kv0 + kBN - 1 > q0) || (win > 0 && kv0 < q0 + kBM - win)) {
                    // visible: lo <= key < hi
                    const int hi = p.causal ? min(n, q0 + row + 1) : n;
                    const int lo = win > 0 ? q0 + row - win + 1 : 0;
#pragma unroll
                    for (int c = 0; c < 128; ++c)
                        if (kv0 + c >= hi || kv0 + c < lo) s[c] = __float_as_uint(-INFINITY);
                }
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
                __syncwarp();
                // a row that has seen no visible key yet (its window starts in a
                // later tile) keeps m_ref = -inf: use 0, so that its masked
                // scores give P = 0 rather than -inf - (-inf)
                const float m_use = (GENERAL && m_ref == -INFINITY) ? 0.0f : m_ref;
                const float2 neg_m = make_float2(-m_use, -m_use);
                const float2 sl2x2 = make_float2(sl2, sl2);
                float2 lr01 = make_float2(0.f, 0.f), lr23 = lr01, le01 = lr01, le23 = lr01;
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
                        const int kq = (c - CH * hh) / 2;
                        if constexpr (BF16) {
                            pk[kq] = pack_bf16x2(p0, p1);
                            pk[kq + 1] = pack_bf16x2(p2, p3);
                            lr01 = add_bf16x2_f32x2(pk[kq], lr01);
                            lr23 = add_bf16x2_f32x2(pk[kq + 1], lr23);
                        } else {
                            pk[kq] = pack_f16x2(p0, p1);
                            pk[kq + 1] = pack_f16x2(p2, p3);
                            lr01 = fadd2(lr01, unpack2<BF16>(pk[kq]));
                            lr23 = fadd2(lr23, unpack2<BF16>(pk[kq + 1]));
                        }
                        le01 = fadd2(le01, make_float2(p0, p1));
                        le23 = fadd2(le23, make_float2(p2, p3));
                    }
                    tmem_st_x16(lane_base + col_s + 16 * hh, pk);
                }
                l_sum += (lr01.x + lr01.y) + (lr23.x + lr23.y);
                l_exact += (le01.x + le01.y) + (le23.x + le23.y);
                // O_x holds this block's P(jx0..j-1) V; warp-uniform rescale
                if (j > jx0 && __any_sync(0xffffffffu, rescale)) {
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
            if (!ok) break;
            // epilogue: O = O~ / l and L = m + ln l, once the block's last P.V
            // of this tile has completed; each thread stores its own row
            const bool got_o = mbar_wait(&o_final[x], nf & 1, abort_flag, p.status, 72);
            if (!__all_sync(0xffffffffu, got_o)) break;
            ++nf;
            tc_fence_after();
            const float inv_l = 1.0f / l_sum;
            const bool in = q0 + row < n;
            // O row r of [B][Hq][N][d] (dense) or [total][Hq][d] (packed); LSE
            // entry li of [B][Hq][N] or [Hq][total]
            size_t r = (size_t)blk.bh * p.N + q0 + row, li = r;
            if (packed) {
                const int h = blk.bh % p.Hq;
                r = (size_t)(row0 + q0 + row) * p.Hq + h;
                li = (size_t)h * p.total + row0 + q0 + row;
            }
            uint8_t *dst = static_cast<uint8_t *>(p.o) + r * (D * 2);
#pragma unroll 1
            for (int c0 = 0; c0 < D; c0 += 32) {
                uint32_t o[32];
                tmem_ld_x32(lane_base + col_o + c0, o);
                tmem_ld_wait_x32(o);
                uint32_t w[16];
#pragma unroll
                for (int c = 0; c < 16; ++c) {
                    const float a0 = __uint_as_float(o[2 * c]) * inv_l;
                    const float a1 = __uint_as_float(o[2 * c + 1]) * inv_l;
                    w[c] = BF16 ? pack_bf16x2(a0, a1) : pack_f16x2(a0, a1);
                }
                if (in) {  // 64 bytes of the row: two whole 32-byte sectors
                    st_global_v8(dst + c0 * 2, w);
                    st_global_v8(dst + c0 * 2 + 32, w + 8);
                }
            }
            if (in) p.lse[li] = (m_ref + log2f(l_exact)) * 0.69314718055994530942f;
            // the next block's first P.V overwrites O_x only after this
            // warpgroup's next p_full arrival, which follows these loads
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
cudaError_t launch_fwd_persist_t(const FwdArgs &a, cudaStream_t st) {
    const bool general = a.window > 0 || a.lay.varlen;
    using L = PersistLayout<D>;
    const CUtensorMapDataType dt = BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    CUtensorMap tq, tk, tv;
    if (!make_tmap_tiles(&tq, a.q, dt, D, a.lay, a.Hq, kBM) || !make_tmap_tiles(&tk, a.k, dt, D, a.lay, a.Hkv, kBN) ||
        !make_tmap_tiles(&tv, a.v, dt, D, a.lay, a.Hkv, kBN))
        return cudaErrorInvalidValue;
    auto kernel = general ? fwd_persist_kernel<D, BF16, true> : fwd_persist_kernel<D, BF16, false>;
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, L::ALLOC);
    if (e != cudaSuccess) return e;
    PersistParams p;
    p.o = a.o;
    p.lse = a.lse;
    p.status = device_status_ptr();
    p.cu_seqlens = a.lay.cu_seqlens;
    p.varlen = a.lay.varlen;
    p.total = a.lay.total;
    p.window = a.window;
    p.Hq = a.Hq;
    p.Hkv = a.Hkv;
    p.N = a.N;
    p.nblk = (a.N + 2 * kBM - 1) / (2 * kBM);
    p.causal = a.causal;
    int dev = 0, sms = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    p.planes = a.B * a.Hq;
    p.group = grid_group_planes(p.planes, p.nblk, sms);
    p.scale_log2 = a.scale * 1.4426950408889634f;
    const long long grid = (long long)p.nblk * a.B * a.Hq;
    kernel<<<dim3((unsigned)grid), dim3(kThreads), L::ALLOC, st>>>(tq, tk, tv, p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd_persist(const FwdArgs &a, cudaStream_t st) {
    if (a.o_f32) return cudaErrorInvalidValue;  // 16-bit output only
    if (reinterpret_cast<uintptr_t>(a.o) & 31u) return cudaErrorInvalidValue;     // 32-byte row stores
    if (a.d == 128) return a.bf16 ? launch_fwd_persist_t<128, true>(a, st) : launch_fwd_persist_t<128, false>(a, st);
    if (a.d == 64) return a.bf16 ? launch_fwd_persist_t<64, true>(a, st) : launch_fwd_persist_t<64, false>(a, st);
    return cudaErrorInvalidValue;
}

}  // namespace fa
