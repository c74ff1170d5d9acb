// fa_bwd_persist.cu -- persistent main kernel of the FlashAttention-2 backward
// for sm_103a (dense layout, bf16 / fp16, d = 64 or 128, causal or not, dQ by
// fp32 atomic reduction).
//
// Same algorithm and per-tile arithmetic as bwd_main_kernel in fa_bwd.cu
// (blog.csdn.net FlashAttention-2 article, 3.1.2 and "parallelism /
// backward": one work item per K/V tile of one key/value head, walking the Q
// tiles of every query head of its group; dV and dK accumulated on chip, dQ
// added into an fp32 accumulator shared by all work items).  What changes is
// the life of a CTA, as in the persistent forward (fa_fwd_persist.cu; the
// FlashAttention-3 summary page names the persistent kernel among its
// remaining optimisations): the grid holds one CTA per work item in the plain
// kernel's L2-grouped, longest-first order, and every CTA that runs keeps
// running, taking the work items of CTAs it cancels before they launch
// (cluster launch control), so items are handed out dynamically in launch
// order with no counter in global memory.  Per CTA, a plain launch pays
// ≈4 µs of set-up, pipeline fill and epilogue plus ≈1.3 µs between CTAs on an
// SM (measured); here the launch gap disappears, and each item's dK/dV
// epilogue (by the softmax warps, stored row by row from registers in whole
// 32-byte sectors) and the atomics of its last dQ tile overlap the next
// item's K/V load.  fa_bwd uses it for short sequences only, where that
// per-CTA cost weighs most.
// Warps, tensor-memory columns and the per-tile MMA order are those of
// bwd_main_kernel; the Q/dO ring positions and all per-tile barrier phases
// carry on across items.
#include "grid_order.cuh"
#include "host_util.h"
#include "ptx.cuh"

namespace fa {

namespace {

constexpr int kBQ = 128;              // query rows per Q tile
constexpr int kBKV = 128;             // key rows per work item (TMEM lanes)
constexpr int kThreads = 576;         // 18 warps
constexpr int kReadoutThreads = 256;  // warps 8-15
constexpr int kSmWarps = 8;           // warps 0-7
constexpr int kNCH = 4;               // 16-query chunks per softmax warp
constexpr int kProducerWarp = 16, kMmaWarp = 17;

template <int D>
struct PBwdLayout {
    static constexpr int NBOX = D / 64;
    static constexpr int TILE_KV = kBKV * D * 2;
    static constexpr int TILE_Q = kBQ * D * 2;
    static constexpr int BOX_KV = kBKV * 128;
    static constexpr int BOX_Q = kBQ * 128;
    static constexpr int QS = 2;  // Q/dO ring depth
    static constexpr int DS_BYTES = kBKV * kBQ * 2;
    static constexpr int DS_BOX = kBKV * 128;
    static constexpr int OFF_K = 0;
    static constexpr int OFF_V = OFF_K + TILE_KV;
    static constexpr int OFF_QD = OFF_V + TILE_KV;  // stage s: Q at +2s*TILE_Q, dO at +(2s+1)*TILE_Q
    static constexpr int OFF_DS = OFF_QD + QS * 2 * TILE_Q;
    static constexpr int OFF_LD = OFF_DS + DS_BYTES;  // stage s: L2[128], D[128]
    static constexpr int OFF_BAR = OFF_LD + QS * 2 * kBQ * 4;
    // kv_full, kv_empty, qd_full[QS], qd_empty[QS], s_full, dp_full, p_ready,
    // ds_ready, dq_full, dq_free, acc_done, drain, ds_half, ds_smem,
    // item_full[2], item_empty[2], clc
    static constexpr int NBAR = 2 + 2 * QS + 10 + 4 + 1;
    static constexpr int OFF_CLC = (OFF_BAR + NBAR * 8 + 15) / 16 * 16;
    static constexpr int OFF_MISC = OFF_CLC + 16;  // item slots [2], TMEM base, abort flag
    static constexpr int BYTES = OFF_MISC + 16;
    static constexpr int SLACK = 512;  // room to align the dynamic shared base up to 1024
    static constexpr int ALLOC = BYTES + SLACK;
    static_assert(ALLOC <= 227 * 1024, "shared memory");
};

struct PBwdParams {
    const float *lse;
    const float *Dvec;
    float *dq_acc;
    void *dk, *dv;
    unsigned int *status;
    int Hq, Hkv, N, nkv, nq;
    int causal;
    int group, planes;  // CTA order (grid_order.cuh): key/value planes per group, B * Hkv
    float scale, scale_log2;
};

constexpr uint32_t kColS = 0, kColDP = 128, kColDQ = 128, kColDV = 256, kColDK = 384;

__device__ __forceinline__ void clc_try_cancel(void *resp, uint64_t *bar) {
    asm volatile(
        "clusterlaunchcontrol.try_cancel.async.shared::cta.mbarrier::complete_tx::bytes.b128 [%0], [%1];" ::"r"(
            smem_u32(resp)),
        "r"(smem_u32(bar))
        : "memory");
}

// The canceled CTA's x index, or -1 if nothing was left to cancel.
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

// The work item an index stands for (the plain kernel's grid order).
struct Item {
    int bg, b, g, kv0, i_start, n_i, n_it;
};

__device__ __forceinline__ Item decode_item(int idx, const PBwdParams &p) {
    Item it;
    int jt;
    grid_decode(idx, p.planes, p.nkv, p.group, it.bg, jt);
    it.b = it.bg / p.Hkv;
    it.g = it.bg - it.b * p.Hkv;
    it.kv0 = jt * kBKV;
    it.i_start = p.causal ? jt : 0;
    it.n_i = p.nq - it.i_start;
    it.n_it = (p.Hq / p.Hkv) * it.n_i;
    return it;
}

template <int D, bool BF16>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_persist_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                       const PBwdParams p) {
    using L = PBwdLayout<D>;
    constexpr int QS = L::QS;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t pad = (1024u - (smem_u32(smem_raw) & 1023u)) & 1023u;
    if (pad > (uint32_t)L::SLACK) {  // uniform across the CTA; nothing started yet
        if (threadIdx.x == 0) record_bad_launch(p.status);
        return;
    }
    uint8_t *smem = smem_raw + pad;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::OFF_BAR);
    uint64_t *kv_full = bars;
    uint64_t *kv_empty = kv_full + 1;
    uint64_t *qd_full = kv_empty + 1;
    uint64_t *qd_empty = qd_full + QS;
    uint64_t *s_full = qd_empty + QS;
    uint64_t *dp_full = s_full + 1;
    uint64_t *p_ready = dp_full + 1;
    uint64_t *ds_ready = p_ready + 1;
    uint64_t *dq_full = ds_ready + 1;
    uint64_t *dq_free = dq_full + 1;
    uint64_t *acc_done = dq_free + 1;
    uint64_t *drain = acc_done + 1;
    uint64_t *ds_half = drain + 1;
    uint64_t *ds_smem = ds_half + 1;
    uint64_t *item_full = ds_smem + 1;    // [2]
    uint64_t *item_empty = item_full + 2;  // [2]
    uint64_t *clc_bar = item_empty + 2;
    void *clc_resp = smem + L::OFF_CLC;
    volatile int *item_slot = reinterpret_cast<volatile int *>(smem + L::OFF_MISC);  // [2]
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L::OFF_MISC + 8);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::OFF_MISC + 12);
    float *ld_smem = reinterpret_cast<float *>(smem + L::OFF_LD);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int G = p.Hq / p.Hkv;

    if (threadIdx.x == 0) {
        mbar_init(kv_full, 1);
        mbar_init(kv_empty, 1);
        for (int s = 0; s < QS; ++s) {
            // 1 arrival with the expected transaction bytes + 32 after L and D
            mbar_init(&qd_full[s], 33);
            mbar_init(&qd_empty[s], 1);
        }
        mbar_init(s_full, 1);
        mbar_init(dp_full, 1);
        mbar_init(p_ready, kSmWarps * 32);
        mbar_init(ds_ready, kSmWarps * 32);
        mbar_init(ds_half, kSmWarps * 32);
        mbar_init(ds_smem, kSmWarps * 32);
        mbar_init(dq_full, 1);
        mbar_init(dq_free, kReadoutThreads);
        mbar_init(acc_done, 1);
        mbar_init(drain, 1);
        for (int x = 0; x < 2; ++x) {
            mbar_init(&item_full[x], 1);
            // the MMA thread + lane 0 of each softmax and read-out warp
            mbar_init(&item_empty[x], 1 + kSmWarps + kReadoutThreads / 32);
        }
        mbar_init(clc_bar, 1);
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

    auto q_stage = [&](int st) { return smem + L::OFF_QD + (2 * st) * L::TILE_Q; };
    auto do_stage = [&](int st) { return smem + L::OFF_QD + (2 * st + 1) * L::TILE_Q; };

    if (warp == kProducerWarp) {
        // ---------------------------------------- TMA producer and scheduler
        int item = blockIdx.x;
        int base = 0;       // Q/dO ring position of the item's first Q tile
        int issued = 0;     // Q/dO ring positions whose copies were issued
        int kv_issued = 0;  // items whose K/V copies were issued (lane 0)
        int clc_n = 0;
        bool clc_pending = false;
        bool ok = true;
        int k = 0;
        if (lane == 0) {
            prefetch_tmap(&tm_q);
            prefetch_tmap(&tm_do);
            prefetch_tmap(&tm_k);
            prefetch_tmap(&tm_v);
        }
        for (;; ++k) {
            // publish the item to the other roles (two slots)
            const int slot = k & 1;
            if (lane == 0) {
                if (k >= 2) ok = mbar_wait(&item_empty[slot], ((k >> 1) - 1) & 1, abort_flag, p.status, 80);
                if (ok) {
                    item_slot[slot] = item;
                    mbar_arrive(&item_full[slot]);
                    if (item >= 0) {
                        mbar_arrive_expect_tx(clc_bar, 16);
                        clc_try_cancel(clc_resp, clc_bar);
                        clc_pending = true;
                    }
                }
            }
            ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
            if (!ok || item < 0) break;
            const Item w = decode_item(item, p);
            // K and V first (once the previous item's last MMAs have read
            // theirs), then the item's Q/dO tiles
            {
                bool okk = true;
                if (lane == 0) {
                    if (k > 0) okk = mbar_wait(kv_empty, (k - 1) & 1, abort_flag, p.status, 81);
                    if (okk) {
                        mbar_arrive_expect_tx(kv_full, 2 * L::TILE_KV);
                        for (int bx = 0; bx < L::NBOX; ++bx) {
                            tma_load_3d(smem + L::OFF_K + bx * L::BOX_KV, &tm_k, kv_full, bx * 64, w.kv0, w.bg);
                            tma_load_3d(smem + L::OFF_V + bx * L::BOX_KV, &tm_v, kv_full, bx * 64, w.kv0, w.bg);
                        }
                        kv_issued = k + 1;
                    }
                }
                okk = __shfl_sync(0xffffffffu, okk ? 1 : 0, 0) != 0;
                if (!okk) break;
            }
            for (int it = 0; it < w.n_it; ++it) {
                const int gi = base + it;  // global ring position
                const int st = gi % QS;
                bool okw = true;
                if (lane == 0 && gi >= QS)
                    okw = mbar_wait(&qd_empty[st], ((gi / QS) + 1) & 1, abort_flag, p.status, 82);
                okw = __shfl_sync(0xffffffffu, okw ? 1 : 0, 0) != 0;
                if (!okw) { ok = false; break; }
                const int h = w.g * G + it / w.n_i;
                const int q_base = (w.i_start + it % w.n_i) * kBQ;
                const int plane = w.b * p.Hq + h;
                if (lane == 0) {
                    mbar_arrive_expect_tx(&qd_full[st], 2 * L::TILE_Q);
                    for (int bx = 0; bx < L::NBOX; ++bx) {
                        tma_load_3d(q_stage(st) + bx * L::BOX_Q, &tm_q, &qd_full[st], bx * 64, q_base, plane);
                        tma_load_3d(do_stage(st) + bx * L::BOX_Q, &tm_do, &qd_full[st], bx * 64, q_base, plane);
                    }
                }
                float *l2s = ld_smem + st * 2 * kBQ;
                float *dsm = l2s + kBQ;
                for (int r = lane; r < kBQ; r += 32) {
                    const int row = q_base + r;
                    const bool in = row < p.N;
                    const size_t li = (size_t)plane * p.N + row;
                    l2s[r] = in ? -p.lse[li] * 1.4426950408889634f : -INFINITY;
                    dsm[r] = in ? p.Dvec[li] : 0.0f;
                }
                mbar_arrive(&qd_full[st]);
                issued = gi + 1;
            }
            if (!ok) break;
            base += w.n_it;
            // the next item: the one whose CTA was canceled, or none
            if (lane == 0) {
                ok = mbar_wait(clc_bar, clc_n & 1, abort_flag, p.status, 83);
                if (ok) {
                    ++clc_n;
                    clc_pending = false;
                    item = clc_result(clc_resp);
                }
            }
            ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
            item = __shfl_sync(0xffffffffu, item, 0);
            if (!ok) break;
        }
        if (lane == 0 && *abort_flag) {
            // let copies and the cancellation request in flight land first
            if (kv_issued > 0) mbar_wait_drain(kv_full, (kv_issued - 1) & 1, 10000000ull);
            for (int t = max(0, issued - QS); t < issued; ++t)
                mbar_wait_drain(&qd_full[t % QS], (t / QS) & 1, 10000000ull);
            if (clc_pending) mbar_wait_drain(clc_bar, clc_n & 1, 10000000ull);
        }
        __syncwarp();
    } else if (warp == kMmaWarp) {
        // ------------------------------------------------------- MMA issuer
        if (lane == 0) {
            constexpr uint32_t fmt = BF16 ? 1u : 0u;
            constexpr uint32_t idesc_sdp = make_idesc(kBKV, kBQ, fmt, false, false);
            constexpr uint32_t idesc_acc = make_idesc(kBKV, D, fmt, false, true);
            constexpr uint32_t idesc_dq = make_idesc(kBKV, kBQ, fmt, true, true);
            const uint64_t k_desc = make_sdesc_sw128(smem_u32(smem + L::OFF_K), 16, 1024);
            const uint64_t v_desc = make_sdesc_sw128(smem_u32(smem + L::OFF_V), 16, 1024);
            const uint64_t kt_desc = make_sdesc_sw128(smem_u32(smem + L::OFF_K), D == 128 ? L::BOX_KV : 0, 1024);
            const uint64_t qk_desc0 = make_sdesc_sw128(smem_u32(q_stage(0)), 16, 1024);
            const uint64_t dok_desc0 = make_sdesc_sw128(smem_u32(do_stage(0)), 16, 1024);
            const uint64_t qm_desc0 = make_sdesc_sw128(smem_u32(q_stage(0)), L::BOX_Q, 1024);
            const uint64_t dom_desc0 = make_sdesc_sw128(smem_u32(do_stage(0)), L::BOX_Q, 1024);
            const uint64_t ds_desc = make_sdesc_sw128(smem_u32(smem + L::OFF_DS), L::DS_BOX, 1024);
            constexpr uint32_t kStage = 2 * L::TILE_Q;

            // S^T of ring position gi -> [0, 128) (s_full)
            auto issue_s = [&](int gi) -> bool {
                const int st = gi % QS;
                if (!mbar_wait(&qd_full[st], (gi / QS) & 1, abort_flag, p.status, 84)) return false;
                tc_fence_after();
                const uint64_t q_desc = sdesc_advance(qk_desc0, st * kStage);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t okv = (kk >> 2) * L::BOX_KV + (kk & 3) * 32;
                    const uint32_t oq = (kk >> 2) * L::BOX_Q + (kk & 3) * 32;
                    mma_f16_ss(tmem + kColS, sdesc_advance(k_desc, okv), sdesc_advance(q_desc, oq), idesc_sdp,
                               kk > 0 ? 1u : 0u);
                }
                mma_commit(s_full);
                return true;
            };
            // dP^T of ring position gi -> [128, 256) (dp_full)
            auto issue_dp = [&](int gi) {
                const uint64_t do_desc = sdesc_advance(dok_desc0, (gi % QS) * kStage);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t okv = (kk >> 2) * L::BOX_KV + (kk & 3) * 32;
                    const uint32_t oq = (kk >> 2) * L::BOX_Q + (kk & 3) * 32;
                    mma_f16_ss(tmem + kColDP, sdesc_advance(v_desc, okv), sdesc_advance(do_desc, oq), idesc_sdp,
                               kk > 0 ? 1u : 0u);
                }
                mma_commit(dp_full);
            };

            int base = 0;  // global ring position of the item's first Q tile
            bool ok = true;
            for (int k = 0; ok; ++k) {
                const int slot = k & 1;
                if (!mbar_wait(&item_full[slot], (k >> 1) & 1, abort_flag, p.status, 85)) break;
                const int item = item_slot[slot];
                mbar_arrive(&item_empty[slot]);
                if (item < 0) break;
                const Item w = decode_item(item, p);
                if (!mbar_wait(kv_full, k & 1, abort_flag, p.status, 86)) break;
                tc_fence_after();
                // the first S^T and dP^T of the item; dP^T overwrites the
                // previous item's last dQ^T once the read-out warps have it
                if (!issue_s(base)) break;
                if (base > 0) {
                    if (!mbar_wait(dq_free, (base - 1) & 1, abort_flag, p.status, 87)) break;
                    tc_fence_after();
                }
                issue_dp(base);
                for (int it = 0; ok && it < w.n_it; ++it) {
                    const int gi = base + it;
                    const int st = gi % QS;
                    const uint64_t qm_desc = sdesc_advance(qm_desc0, st * kStage);
                    const uint64_t dom_desc = sdesc_advance(dom_desc0, st * kStage);
                    const uint32_t acc_first = it > 0 ? 1u : 0u;
                    // dV += P^T dO (A = P^T from tensor memory)
                    if (!mbar_wait(p_ready, gi & 1, abort_flag, p.status, 88)) { ok = false; break; }
                    tc_fence_after();
#pragma unroll
                    for (int kk = 0; kk < kBQ / 16; ++kk)
                        mma_f16_ts(tmem + kColDV, tmem + kColS + kk * 16, sdesc_advance(dom_desc, kk * 2048),
                                   idesc_acc, kk > 0 ? 1u : acc_first);
                    // dK += dS^T Q in two sets of 16-query steps (the first two
                    // chunks of every softmax warp as soon as they are written)
                    auto issue_dk = [&](bool first) {
#pragma unroll
                        for (int kk = 0; kk < kBQ / 16; ++kk)
                            if (((kk & 3) < 2) == first)
                                mma_f16_ts(tmem + kColDK, tmem + kColS + kk * 16 + 8, sdesc_advance(qm_desc, kk * 2048),
                                           idesc_acc, kk > 0 ? 1u : acc_first);
                    };
                    if (!mbar_wait(ds_half, gi & 1, abort_flag, p.status, 89)) { ok = false; break; }
                    tc_fence_after();
                    issue_dk(true);
                    if (!mbar_wait(ds_ready, gi & 1, abort_flag, p.status, 90)) { ok = false; break; }
                    tc_fence_after();
                    issue_dk(false);
                    mma_commit(&qd_empty[st]);  // dK is the last reader of this Q/dO stage
                    // S^T of the next Q tile of this item (not the next item's:
                    // its K and V arrive only once this item's MMAs are done)
                    if (it + 1 < w.n_it && !issue_s(gi + 1)) { ok = false; break; }
                    // dQ^T = K^T dS^T -> [128, 256)
                    if (!mbar_wait(ds_smem, gi & 1, abort_flag, p.status, 91)) { ok = false; break; }
                    tc_fence_after();
#pragma unroll
                    for (int kk = 0; kk < kBKV / 16; ++kk)
                        mma_f16_ss(tmem + kColDQ, sdesc_advance(kt_desc, kk * 2048), sdesc_advance(ds_desc, kk * 2048),
                                   idesc_dq, kk > 0 ? 1u : 0u);
                    mma_commit(dq_full);
                    if (it + 1 < w.n_it) {
                        if (!mbar_wait(dq_free, gi & 1, abort_flag, p.status, 92)) { ok = false; break; }
                        tc_fence_after();
                        issue_dp(gi + 1);
                    }
                }
                if (!ok) break;
                base += w.n_it;
                mma_commit(kv_empty);  // K and V were last read by the dQ^T just issued
                mma_commit(acc_done);  // dV and dK of this item are complete
            }
            mma_commit(drain);
            mbar_wait_drain(drain, 0, 100000000ull);
        }
        __syncwarp();
    } else if (warp < kSmWarps) {
        // --------------------------- warps 0-7: softmax (P^T, dS^T), epilogue
        const int hf = warp >> 2;
        const int q0w = hf * 16 * kNCH;
        const int quarter = warp & 3;
        const int c = quarter * 32 + lane;  // key row == TMEM lane
        const uint32_t lane_base = tmem + ((uint32_t)(quarter * 32) << 16);
        const float2 sl2 = make_float2(p.scale_log2, p.scale_log2);
        int base = 0;
        bool ok = true;
        for (int k = 0; ok; ++k) {
            const int slot = k & 1;
            const bool got = mbar_wait(&item_full[slot], (k >> 1) & 1, abort_flag, p.status, 93);
            if (!__all_sync(0xffffffffu, got)) break;
            const int item = item_slot[slot];
            __syncwarp();
            if (lane == 0) mbar_arrive(&item_empty[slot]);
            if (item < 0) break;
            const Item w = decode_item(item, p);
            const int kv = w.kv0 + c;
            const bool kv_oob = kv >= p.N;  // a zero-filled key row: P = 0
            for (int it = 0; it < w.n_it; ++it) {
                const int gi = base + it;
                const int st = gi % QS;
                const bool w1 = mbar_wait(s_full, gi & 1, abort_flag, p.status, 94);
                const bool w2 = w1 && mbar_wait(&qd_full[st], (gi / QS) & 1, abort_flag, p.status, 95);
                if (!__all_sync(0xffffffffu, w2)) { ok = false; break; }
                tc_fence_after();
                const int q_base = (w.i_start + it % w.n_i) * kBQ;
                const bool diag = p.causal && (q_base + q0w < w.kv0 + kBKV);
                const float *ldst = ld_smem + st * 2 * kBQ;
                // ---- phase 1: P^T (16-bit pairs), kept in registers for phase 2
                uint32_t pp[kNCH][8];
                uint32_t sv[32];
#pragma unroll
                for (int ch = 0; ch < kNCH; ++ch) {
                    const int qc = q0w + ch * 16;
                    const int q_first = q_base + qc;
                    if ((ch & 1) == 0) {
                        tmem_ld_x32(lane_base + kColS + qc, sv);
                        tmem_ld_wait_x32(sv);
                    }
                    const uint32_t *s = sv + 16 * (ch & 1);
                    float nl[16];
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const float4 f = *reinterpret_cast<const float4 *>(ldst + qc + 4 * q);
                        nl[4 * q] = f.x;
                        nl[4 * q + 1] = f.y;
                        nl[4 * q + 2] = f.z;
                        nl[4 * q + 3] = f.w;
                    }
#pragma unroll
                    for (int r = 0; r < 16; r += 2) {
                        const float2 x = ffma2(make_float2(__uint_as_float(s[r]), __uint_as_float(s[r + 1])), sl2,
                                               make_float2(nl[r], nl[r + 1]));
                        float p0 = ex2_approx(x.x);
                        float p1 = ex2_approx(x.y);
                        if (diag) {  // causal: key kv is visible to query q iff kv <= q
                            if (kv > q_first + r) p0 = 0.0f;
                            if (kv > q_first + r + 1) p1 = 0.0f;
                        }
                        pp[ch][r / 2] = BF16 ? pack_bf16x2(p0, p1) : pack_f16x2(p0, p1);
                    }
                    if (kv_oob) {
#pragma unroll
                        for (int r = 0; r < 8; ++r) pp[ch][r] = 0u;
                    }
                    __syncwarp();
                    tmem_st_x8(lane_base + kColS + qc, pp[ch]);
                }
                tmem_st_wait();
                tc_fence_before();
                mbar_arrive(p_ready);
                // ---- phase 2: dS^T = P^T o (dP^T - D), from the rounded P^T
                const bool w3 = mbar_wait(dp_full, gi & 1, abort_flag, p.status, 96);
                if (!__all_sync(0xffffffffu, w3)) { ok = false; break; }
                tc_fence_after();
                uint8_t *ds_row = smem + L::OFF_DS + hf * L::DS_BOX + c * 128;
                uint32_t dpv[2][16];  // dP^T one chunk at a time, loaded one chunk ahead
                uint32_t ddk[kNCH][8];
                tmem_ld_x16(lane_base + kColDP + q0w, dpv[0]);
#pragma unroll
                for (int ch = 0; ch < kNCH; ++ch) {
                    const int qc = q0w + ch * 16;
                    tmem_ld_wait_x16(dpv[ch & 1]);  // the only load outstanding
                    if (ch + 1 < kNCH) tmem_ld_x16(lane_base + kColDP + qc + 16, dpv[(ch + 1) & 1]);
                    const uint32_t *dp = dpv[ch & 1];
                    float dv_[16];
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const float4 f = *reinterpret_cast<const float4 *>(ldst + kBQ + qc + 4 * q);
                        dv_[4 * q] = f.x;
                        dv_[4 * q + 1] = f.y;
                        dv_[4 * q + 2] = f.z;
                        dv_[4 * q + 3] = f.w;
                    }
                    uint32_t dd[8];
#pragma unroll
                    for (int r = 0; r < 16; r += 2) {
                        const float2 pv = unpack2<BF16>(pp[ch][r / 2]);
                        const float2 t = fsub2(make_float2(__uint_as_float(dp[r]), __uint_as_float(dp[r + 1])),
                                               make_float2(dv_[r], dv_[r + 1]));
                        const float2 ds = fmul2(pv, t);
                        dd[r / 2] = BF16 ? pack_bf16x2(ds.x, ds.y) : pack_f16x2(ds.x, ds.y);
                    }
                    __syncwarp();
                    tmem_st_x8(lane_base + kColS + qc + 8, dd);
                    if (ch == kNCH / 2 - 1) {
                        tmem_st_wait();
                        tc_fence_before();
                        mbar_arrive(ds_half);
                    }
#pragma unroll
                    for (int r = 0; r < 8; ++r) ddk[ch][r] = dd[r];
                }
                tmem_st_wait();
                tc_fence_before();
                mbar_arrive(ds_ready);
#pragma unroll
                for (int ch = 0; ch < kNCH; ++ch)
#pragma unroll
                    for (int q = 0; q < 2; ++q)
                        *reinterpret_cast<uint4 *>(ds_row + (((2 * ch + q) ^ (c & 7)) << 4)) =
                            make_uint4(ddk[ch][4 * q], ddk[ch][4 * q + 1], ddk[ch][4 * q + 2], ddk[ch][4 * q + 3]);
                fence_proxy_async_smem();
                mbar_arrive(ds_smem);
            }
            if (!ok) break;
            base += w.n_it;
            // epilogue: dV (warps 0-3) or dK (warps 4-7) of this item, each
            // thread storing its own key row from registers; the next item's
            // first dV / dK MMA overwrites these columns only after this
            // warpgroup's next p_ready / ds_half arrival
            const bool got_acc = mbar_wait(acc_done, k & 1, abort_flag, p.status, 97);
            if (!__all_sync(0xffffffffu, got_acc)) break;
            tc_fence_after();
            const uint32_t col = hf == 0 ? kColDV : kColDK;
            const float f = hf == 0 ? 1.0f : p.scale;
            uint8_t *dst = static_cast<uint8_t *>(hf == 0 ? p.dv : p.dk) + ((size_t)w.bg * p.N + kv) * (D * 2);
#pragma unroll 1
            for (int c0 = 0; c0 < D; c0 += 32) {
                uint32_t o[32];
                tmem_ld_x32(lane_base + col + c0, o);
                tmem_ld_wait_x32(o);
                uint32_t u[16];
#pragma unroll
                for (int x = 0; x < 16; ++x) {
                    const float a0 = __uint_as_float(o[2 * x]) * f;
                    const float a1 = __uint_as_float(o[2 * x + 1]) * f;
                    u[x] = BF16 ? pack_bf16x2(a0, a1) : pack_f16x2(a0, a1);
                }
                if (!kv_oob) {  // 64 bytes of the row: two whole 32-byte sectors
                    st_global_v8(dst + c0 * 2, u);
                    st_global_v8(dst + c0 * 2 + 32, u + 8);
                }
            }
        }
        __syncwarp();
    } else {
        // ------------------- warps 8-15: dQ^T read-out and atomic reduction
        const int hf = (warp - 8) >> 2;
        const int quarter = warp & 3;
        const int t = quarter * 32 + lane;
        const uint32_t lane_base = tmem + ((uint32_t)(quarter * 32) << 16);
        int base = 0;
        for (int k = 0;; ++k) {
            const int slot = k & 1;
            const bool got = mbar_wait(&item_full[slot], (k >> 1) & 1, abort_flag, p.status, 98);
            if (!__all_sync(0xffffffffu, got)) break;
            const int item = item_slot[slot];
            __syncwarp();
            if (lane == 0) mbar_arrive(&item_empty[slot]);
            if (item < 0) break;
            const Item w = decode_item(item, p);
            bool ok = true;
            for (int it = 0; it < w.n_it; ++it) {
                const int gi = base + it;
                const bool g2 = mbar_wait(dq_full, gi & 1, abort_flag, p.status, 99);
                if (!__all_sync(0xffffffffu, g2)) { ok = false; break; }
                tc_fence_after();
                uint32_t v[64];
                tmem_ld_x32(lane_base + kColDQ + hf * 64, v);
                tmem_ld_x32(lane_base + kColDQ + hf * 64 + 32, v + 32);
                tmem_ld_wait_x32(v);
                tmem_ld_wait_x32(v + 32);
                tc_fence_before();
                mbar_arrive(dq_free);
                const int h = w.g * G + it / w.n_i;
                const int q_first = (w.i_start + it % w.n_i) * kBQ + hf * 64;
                const int rows = min(64, p.N - q_first);
                if (t < D) {
                    float *dst = p.dq_acc + ((size_t)(w.b * p.Hq + h) * p.N + q_first) * D + t;
#pragma unroll
                    for (int r = 0; r < 64; ++r)
                        if (r < rows) atomicAdd(dst + (size_t)r * D, __uint_as_float(v[r]));
                }
            }
            if (!ok) break;
            base += w.n_it;
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
cudaError_t launch_t(const BwdArgs &a, cudaStream_t st) {
    using L = PBwdLayout<D>;
    const CUtensorMapDataType dt = BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    CUtensorMap tq, tk, tv, tdo;
    if (!make_tmap_tiles(&tq, a.q, dt, D, a.lay, a.Hq, kBQ) || !make_tmap_tiles(&tdo, a.dO, dt, D, a.lay, a.Hq, kBQ) ||
        !make_tmap_tiles(&tk, a.k, dt, D, a.lay, a.Hkv, kBKV) || !make_tmap_tiles(&tv, a.v, dt, D, a.lay, a.Hkv, kBKV))
        return cudaErrorInvalidValue;
    auto kernel = bwd_persist_kernel<D, BF16>;
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, L::ALLOC);
    if (e != cudaSuccess) return e;
    PBwdParams p;
    p.lse = a.lse;
    p.Dvec = a.D;
    p.dq_acc = a.dq_acc;
    p.dk = a.dk;
    p.dv = a.dv;
    p.status = device_status_ptr();
    p.Hq = a.Hq;
    p.Hkv = a.Hkv;
    p.N = a.N;
    p.nkv = (a.N + kBKV - 1) / kBKV;
    p.nq = (a.N + kBQ - 1) / kBQ;
    p.causal = a.causal;
    p.scale = a.scale;
    p.scale_log2 = a.scale * 1.4426950408889634f;
    int dev = 0, sms = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    p.planes = a.B * a.Hkv;
    p.group = grid_group_planes(p.planes, p.nkv, sms);
    const long long grid = (long long)p.nkv * a.B * a.Hkv;
    kernel<<<dim3((unsigned)grid), dim3(kThreads), L::ALLOC, st>>>(tq, tk, tv, tdo, p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_persist_main(const BwdArgs &a, cudaStream_t st) {
    if (a.window > 0 || a.lay.varlen || !a.dq_acc) return cudaErrorInvalidValue;  // dense, atomic dQ only
    if ((reinterpret_cast<uintptr_t>(a.dk) | reinterpret_cast<uintptr_t>(a.dv)) & 31u)
        return cudaErrorInvalidValue;  // 32-byte row stores
    if (a.d == 128) return a.bf16 ? launch_t<128, true>(a, st) : launch_t<128, false>(a, st);
    if (a.d == 64) return a.bf16 ? launch_t<64, true>(a, st) : launch_t<64, false>(a, st);
    return cudaErrorInvalidValue;
}

}  // namespace fa
