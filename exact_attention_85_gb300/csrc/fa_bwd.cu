// fa_bwd.cu -- FlashAttention-2 backward for sm_103a (bf16 / fp16, d = 64, 128).
//
// Algorithm (blog.csdn.net FlashAttention-2 article, 3.1.2 and "parallelism /
// backward"; "6.2 FlashAttention V2 chi tiet", section 7): only L and
// D = rowsum(dO o O) are used; D comes from a separate preprocessing kernel;
// one CTA owns a K/V column block j and walks every Q tile i, recomputing
// S = Q_i K_j^T and P = exp(S - L_i), accumulating dV_j += P^T dO_i and
// dK_j += dS^T Q_i on chip, and adding dQ_i += dS K_j into an fp32 dQ
// accumulator shared by all CTAs (atomic addition).  Grouped-query heads: the
// CTA of key/value head g walks the Q tiles of all query heads of its group,
// so dK/dV are summed over the group before they are stored (MQA/GQA
// paragraph of the blog.csdn.net page).
//
// Kernels:
//   bwd_pre_kernel   D = rowsum(dO o O) (fp32) and dQacc = 0     (HBM bound)
//   bwd_main_kernel  the K/V-tile loop below                     (tensor bound)
//   bwd_dq_kernel    dQ = scale * dQacc, converted to the element type
// and, for the deterministic two-pass variant, bwd_pre_kernel (D only),
// bwd_main_kernel without its dQ part, then bwd_dq_pass_kernel (one CTA per
// Q tile, dQ summed on chip in a fixed order; described at the kernel).
//
// Main kernel, one CTA per (128-key tile, key/value head, batch); Q tiles of
// 128 rows, so every MMA is 128 x 128 (full tensor-core rate; at 64 columns the
// shared-memory operand traffic caps the rate near two thirds).  Tensor
// memory (512 columns, fp32, lane = key row unless noted):
//   [0, 128)   S^T = K_j Q_i^T    -> then, per 16-query chunk m, P^T in
//              [16 m, 16 m + 8) and dS^T in [16 m + 8, 16 m + 16) (16-bit pairs)
//   [128, 256) dP^T = V_j dO_i^T  -> then dQ_i^T = K_j^T dS_i^T (lane = head-dim index)
//   [256, 256 + d) dV_j,  [384, 384 + d) dK_j  (accumulated over all Q tiles)
// P^T and dS^T stay in tensor memory as the A operands of dV += P^T dO and
// dK += dS^T Q; dS^T is also written to shared memory as the B operand of
// dQ^T = K^T dS^T.  Per Q tile: MMA S^T -> softmax phase 1 (P^T) while the
// tensor cores compute dP^T -> MMA dV += P^T dO while softmax phase 2 forms
// dS^T -> MMA dK (the steps of each warp's first two query chunks as soon
// as those are written), then the next tile's S^T (the softmax warps start on
// it while the tensor cores go on), then dQ^T (once the softmax warps have
// also copied dS^T to shared memory) -> read-out warps copy dQ^T out of
// tensor memory (which frees the columns for the next dP^T) and add it into
// dQacc with fp32 atomic reductions (one 128-byte line per warp and query
// row) while the softmax warps work on the next tile.
// Warps: 0-7 softmax (then 0-3 store dV, 4-7 store dK), 8-15 dQ read-out
// (softmax too when the kernel runs without its dQ part), 16 TMA producer
// (Q / dO through a 2-deep ring), 17 MMA issuer + TMEM owner.
#include "grid_order.cuh"
#include "host_util.h"
#include "ptx.cuh"

namespace fa {

namespace {

constexpr int kBQ = 128;       // query rows per Q tile
constexpr int kBKV = 128;      // key rows per CTA (TMEM lanes)
constexpr int kThreads = 576;  // 18 warps
constexpr int kReadoutThreads = 256;  // warps 8-15
constexpr int kProducerWarp = 16, kMmaWarp = 17;

template <int D>
struct BwdLayout {
    static constexpr int NBOX = D / 64;
    static constexpr int TILE_KV = kBKV * D * 2;  // K or V tile, bytes
    static constexpr int TILE_Q = kBQ * D * 2;    // Q or dO tile
    static constexpr int BOX_KV = kBKV * 128;     // one 64-column box of a K/V tile
    static constexpr int BOX_Q = kBQ * 128;       // one 64-column box of a Q/dO tile
    static constexpr int QS = 2;                  // Q/dO ring depth
    static constexpr int DS_BYTES = kBKV * kBQ * 2;  // dS^T: two 64-query boxes
    static constexpr int DS_BOX = kBKV * 128;
    static constexpr int OFF_K = 0;
    static constexpr int OFF_V = OFF_K + TILE_KV;
    static constexpr int OFF_QD = OFF_V + TILE_KV;  // stage s: Q at +2s*TILE_Q, dO at +(2s+1)*TILE_Q
    static constexpr int OFF_DS = OFF_QD + QS * 2 * TILE_Q;
    static constexpr int OFF_LD = OFF_DS + DS_BYTES;  // stage s: L2[128], D[128]
    static constexpr int OFF_BAR = OFF_LD + QS * 2 * kBQ * 4;
    // kv_full, qd_full[QS], qd_empty[QS], s_full, dp_full, p_ready, ds_ready,
    // dq_full, dq_free, acc_done, drain, ds_half, ds_smem
    static constexpr int NBAR = 1 + 2 * QS + 6 + 4;
    static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
    static constexpr int BYTES = OFF_MISC + 16;
    static constexpr int SLACK = 512;  // room to align the dynamic shared base up to 1024
    static constexpr int ALLOC = BYTES + SLACK;
    static_assert(TILE_Q >= TILE_KV, "an output tile must fit in one Q (or dO) buffer");
};

struct BwdParams {
    const float *lse;
    const float *Dvec;
    float *dq_acc;
    void *dk, *dv;           // packed layout: stored row by row
    unsigned int *status;
    const int *cu_seqlens;   // packed layout: sequence b is rows cu[b] .. cu[b+1]-1
    int varlen, total;
    int Hq, Hkv, N, nkv, nq;
    int causal;
    int window;  // > 0: query r sees keys r - window + 1 .. r only
    int group;   // key/value planes per CTA-order group (grid_order.cuh)
    float scale, scale_log2;
};

// tensor-memory columns
constexpr uint32_t kColS = 0, kColDP = 128, kColDQ = 128, kColDV = 256, kColDK = 384;

// DQ = false builds the first pass of the deterministic two-pass backward:
// only dK and dV, no dQ^T MMA, no dS in shared memory, no atomics.
// GENERAL = false compiles the sliding window and the packed layout out.
template <int D, bool BF16, bool DQ, bool GENERAL>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_main_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                    const __grid_constant__ CUtensorMap tm_dk, const __grid_constant__ CUtensorMap tm_dv,
                    const BwdParams p) {
    using L = BwdLayout<D>;
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
    uint64_t *qd_full = bars + 1;
    uint64_t *qd_empty = qd_full + QS;
    uint64_t *s_full = qd_empty + QS;
    uint64_t *dp_full = s_full + 1;
    uint64_t *p_ready = dp_full + 1;
    uint64_t *ds_ready = p_ready + 1;
    uint64_t *dq_full = ds_ready + 1;
    uint64_t *dq_free = dq_full + 1;
    uint64_t *acc_done = dq_free + 1;
    uint64_t *drain = acc_done + 1;
    uint64_t *ds_half = drain + 1;    // dS^T of every warp's first two query chunks is in TMEM
    uint64_t *ds_smem = ds_half + 1;  // dS^T is in shared memory (the B operand of dQ^T)
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L::OFF_MISC);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::OFF_MISC + 4);
    float *ld_smem = reinterpret_cast<float *>(smem + L::OFF_LD);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int win = GENERAL ? p.window : 0;
    const bool packed = GENERAL && p.varlen;
    // without the dQ part the read-out warps 8-15 join the softmax: 16 warps,
    // 32 query columns each instead of 8 warps of 64
    constexpr int kSmWarps = DQ ? 8 : 16;
    constexpr int kNCH = DQ ? 4 : 2;  // 16-query chunks per softmax warp

    // CTA order: key/value planes in L2-sized groups; the first K/V tiles of
    // a causal plane visit the most Q tiles and go first
    int bg, jt;  // bg = batch * Hkv + g
    grid_decode(blockIdx.x, (int)(gridDim.x / p.nkv), p.nkv, p.group, bg, jt);
    const int b = bg / p.Hkv;
    const int g = bg - b * p.Hkv;
    const int G = p.Hq / p.Hkv;
    const int kv0 = jt * kBKV;
    // rows of this sequence (packed layout: rows row0 .. row0 + N - 1 of the
    // token-major tensors)
    int N = p.N, row0 = 0;
    if (packed) {
        row0 = p.cu_seqlens[b];
        N = p.cu_seqlens[b + 1] - row0;
        if (N < 0 || N > p.N || row0 < 0 || row0 + N > p.total) {
            if (threadIdx.x == 0 && jt == 0) record_bad_args(p.status);
            return;  // uniform across the CTA, nothing started yet
        }
    }
    if (kv0 >= N) return;  // key tile past the end of a shorter sequence
    const int nq = (N + kBQ - 1) / kBQ;
    const int i_start = p.causal ? jt : 0;  // first Q tile with a row >= kv0 (equal tile sizes)
    // with a sliding window of W keys the last query row that sees any key of
    // this tile is kv0 + 127 + W - 1; later Q tiles are skipped
    const int i_end = win > 0 ? min(nq, (kv0 + kBKV + win - 2) / kBQ + 1) : nq;
    const int n_i = i_end - i_start;
    const int n_it = G * n_i;

    if (threadIdx.x == 0) {
        mbar_init(kv_full, 1);
        for (int s = 0; s < QS; ++s) {
            // 1 arrival with the expected transaction bytes (lane 0, before the
            // copies) + 32 arrivals after the lanes have written L and D
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
        // ------------------------------------------------------ TMA producer
        if (lane == 0) {
            prefetch_tmap(&tm_q);
            prefetch_tmap(&tm_do);
            mbar_arrive_expect_tx(kv_full, 2 * L::TILE_KV);
            for (int bx = 0; bx < L::NBOX; ++bx) {
                const int c1 = packed ? g : kv0, c2 = packed ? row0 + kv0 : bg;
                tma_load_3d(smem + L::OFF_K + bx * L::BOX_KV, &tm_k, kv_full, bx * 64, c1, c2);
                tma_load_3d(smem + L::OFF_V + bx * L::BOX_KV, &tm_v, kv_full, bx * 64, c1, c2);
            }
        }
        int it = 0;
        for (; it < n_it; ++it) {
            const int st = it % QS;
            bool ok = true;
            if (lane == 0 && it >= QS)
                ok = mbar_wait(&qd_empty[st], ((it / QS) + 1) & 1, abort_flag, p.status, 21);
            ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
            if (!ok) break;
            const int h = g * G + it / n_i;
            const int q_base = (i_start + it % n_i) * kBQ;
            const int plane = b * p.Hq + h;
            if (lane == 0) {
                // tensor copies first, so their latency overlaps the L / D loads
                mbar_arrive_expect_tx(&qd_full[st], 2 * L::TILE_Q);
                const int c1 = packed ? h : q_base, c2 = packed ? row0 + q_base : plane;
                for (int bx = 0; bx < L::NBOX; ++bx) {
                    tma_load_3d(q_stage(st) + bx * L::BOX_Q, &tm_q, &qd_full[st], bx * 64, c1, c2);
                    tma_load_3d(do_stage(st) + bx * L::BOX_Q, &tm_do, &qd_full[st], bx * 64, c1, c2);
                }
            }
            float *l2s = ld_smem + st * 2 * kBQ;
            float *dsm = l2s + kBQ;
            for (int r = lane; r < kBQ; r += 32) {
                const int row = q_base + r;
                const bool in = row < N;
                const size_t li = packed ? (size_t)h * p.total + row0 + row : (size_t)plane * N + row;
                // stored negated in log2 units; rows past N get -inf, so P = 0
                l2s[r] = in ? -p.lse[li] * 1.4426950408889634f : -INFINITY;
                dsm[r] = in ? p.Dvec[li] : 0.0f;
            }
            mbar_arrive(&qd_full[st]);  // releases this lane's L / D writes
        }
        if (lane == 0 && *abort_flag) {
            // let copies already in flight land before the CTA exits
            mbar_wait_drain(kv_full, 0, 10000000ull);
            for (int t = max(0, it - QS); t < it; ++t)
                mbar_wait_drain(&qd_full[t % QS], (t / QS) & 1, 10000000ull);
        }
        __syncwarp();
    } else if (warp == kMmaWarp) {
        // ------------------------------------------------------- MMA issuer
        if (lane == 0) {
            constexpr uint32_t fmt = BF16 ? 1u : 0u;
            constexpr uint32_t idesc_sdp = make_idesc(kBKV, kBQ, fmt, false, false);  // K-major both
            constexpr uint32_t idesc_acc = make_idesc(kBKV, D, fmt, false, true);     // A tmem, B MN-major
            constexpr uint32_t idesc_dq = make_idesc(kBKV, kBQ, fmt, true, true);     // A, B MN-major
            // one descriptor per operand tile; steps are derived by sdesc_advance
            const uint64_t k_desc = make_sdesc_sw128(smem_u32(smem + L::OFF_K), 16, 1024);  // K-major
            const uint64_t v_desc = make_sdesc_sw128(smem_u32(smem + L::OFF_V), 16, 1024);
            // K^T as the MN-major A of dQ^T; for d = 64 the second 64-row half of
            // A repeats the first (LBO 0) and those rows are never read out
            const uint64_t kt_desc = make_sdesc_sw128(smem_u32(smem + L::OFF_K), D == 128 ? L::BOX_KV : 0, 1024);
            const uint64_t qk_desc0 = make_sdesc_sw128(smem_u32(q_stage(0)), 16, 1024);          // K-major
            const uint64_t dok_desc0 = make_sdesc_sw128(smem_u32(do_stage(0)), 16, 1024);
            const uint64_t qm_desc0 = make_sdesc_sw128(smem_u32(q_stage(0)), L::BOX_Q, 1024);    // MN-major
            const uint64_t dom_desc0 = make_sdesc_sw128(smem_u32(do_stage(0)), L::BOX_Q, 1024);
            // dS^T rows of 128 queries = two 64-query boxes (MN-major B, LBO = box stride)
            const uint64_t ds_desc = make_sdesc_sw128(smem_u32(smem + L::OFF_DS), L::DS_BOX, 1024);
            constexpr uint32_t kStage = 2 * L::TILE_Q;  // bytes between Q/dO stages
            bool ok = mbar_wait(kv_full, 0, abort_flag, p.status, 22);

            // S^T = K_j Q_t^T -> [0, 128) (commit s_full), and dP^T = V_j dO_t^T
            // -> [128, 256) (commit dp_full): the softmax warps start on P^T as
            // soon as S^T is there, while the tensor cores compute dP^T
            auto issue_s = [&](int t) -> bool {
                const int st = t % QS;
                if (!mbar_wait(&qd_full[st], (t / QS) & 1, abort_flag, p.status, 23)) return false;
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
            auto issue_dp = [&](int t) {
                const uint64_t do_desc = sdesc_advance(dok_desc0, (t % QS) * kStage);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t okv = (kk >> 2) * L::BOX_KV + (kk & 3) * 32;
                    const uint32_t oq = (kk >> 2) * L::BOX_Q + (kk & 3) * 32;
                    mma_f16_ss(tmem + kColDP, sdesc_advance(v_desc, okv), sdesc_advance(do_desc, oq), idesc_sdp,
                               kk > 0 ? 1u : 0u);
                }
                mma_commit(dp_full);
            };

            if (ok) ok = issue_s(0);
            if (ok) issue_dp(0);
            for (int it = 0; ok && it < n_it; ++it) {
                const int st = it % QS;
                const uint64_t qm_desc = sdesc_advance(qm_desc0, st * kStage);
                const uint64_t dom_desc = sdesc_advance(dom_desc0, st * kStage);
                const uint32_t acc_first = it > 0 ? 1u : 0u;
                // dV_j += P^T dO_i as soon as P^T is written (the softmax warps
                // compute dS^T meanwhile).  A from tensor memory: 16 queries = 8
                // packed columns per step; queries 16 m .. 16 m + 15 have P^T at
                // columns 16 m .. + 7 and dS^T at 16 m + 8 .. + 15.
                if (!mbar_wait(p_ready, it & 1, abort_flag, p.status, 30)) { ok = false; break; }
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < kBQ / 16; ++kk)
                    mma_f16_ts(tmem + kColDV, tmem + kColS + kk * 16, sdesc_advance(dom_desc, kk * 2048), idesc_acc,
                               kk > 0 ? 1u : acc_first);
                // dK_j += dS^T Q_i (A from tensor memory, as for dV), as two sets
                // of 16-query steps: those with (step mod 4) < 2 -- with dQ,
                // the first two chunks of every softmax warp, issued as soon
                // as they are written (ds_half) so that they run during the
                // rest of the second phase -- then the others.  Without dQ the
                // same order is kept (one wait), so that both variants sum dK
                // identically.
                auto issue_dk = [&](bool first) {
#pragma unroll
                    for (int kk = 0; kk < kBQ / 16; ++kk)
                        if (((kk & 3) < 2) == first)
                            mma_f16_ts(tmem + kColDK, tmem + kColS + kk * 16 + 8, sdesc_advance(qm_desc, kk * 2048),
                                       idesc_acc, kk > 0 ? 1u : acc_first);
                };
                if constexpr (DQ) {
                    if (!mbar_wait(ds_half, it & 1, abort_flag, p.status, 32)) { ok = false; break; }
                    tc_fence_after();
                    issue_dk(true);
                }
                if (!mbar_wait(ds_ready, it & 1, abort_flag, p.status, 24)) { ok = false; break; }
                tc_fence_after();
                if constexpr (!DQ) issue_dk(true);
                issue_dk(false);
                mma_commit(&qd_empty[st]);  // dK is the last reader of this Q/dO stage
                // S^T of the next tile overwrites P^T, dS^T (read by the MMAs just
                // issued, which run first): issued before dQ^T so that the
                // softmax warps start on the next tile one GEMM earlier
                if (it + 1 < n_it && !issue_s(it + 1)) { ok = false; break; }
                // dQ_i^T = K_j^T dS_i^T -> [128, 256) (lane = head-dim index);
                // 16 keys = 16 rows = 2048 bytes of both operands per step
                if constexpr (DQ) {
                    if (!mbar_wait(ds_smem, it & 1, abort_flag, p.status, 33)) { ok = false; break; }
                    tc_fence_after();
#pragma unroll
                    for (int kk = 0; kk < kBKV / 16; ++kk)
                        mma_f16_ss(tmem + kColDQ, sdesc_advance(kt_desc, kk * 2048),
                                   sdesc_advance(ds_desc, kk * 2048), idesc_dq, kk > 0 ? 1u : 0u);
                    mma_commit(dq_full);
                }
                if (it + 1 < n_it) {
                    // dP^T of the next tile overwrites dQ^T, read out once dq_free flips
                    if constexpr (DQ) {
                        if (!mbar_wait(dq_free, it & 1, abort_flag, p.status, 25)) { ok = false; break; }
                        tc_fence_after();
                    }
                    issue_dp(it + 1);
                }
            }
            if (ok) mma_commit(acc_done);
            // every MMA issued above has completed once `drain` flips
            mma_commit(drain);
            mbar_wait_drain(drain, 0, 100000000ull);
        }
        __syncwarp();
    } else if (warp < kSmWarps) {
        // -------------------- warps 0-7 (0-15 without dQ): softmax (P^T, dS^T)
        // Warp w owns key rows 32 (w % 4) .. + 31 (its TMEM lane quarter) and
        // query columns q0w .. q0w + 16 kNCH - 1 (q0w = 16 kNCH (w / 4)), in
        // chunks of 16 (two per tensor-memory load).
        // Two phases per Q tile: P^T from S^T (then p_ready, so dV += P^T dO
        // runs), then dS^T = P^T o (dP^T - D) once dP^T is there (ds_ready).
        const int hf = warp >> 2;  // query slice; dV (0) or dK (1) in the epilogue
        const int q0w = hf * 16 * kNCH;
        const int quarter = warp & 3;
        const int c = quarter * 32 + lane;  // key row == TMEM lane
        const uint32_t lane_base = tmem + ((uint32_t)(quarter * 32) << 16);
        const float2 sl2 = make_float2(p.scale_log2, p.scale_log2);
        const int kv = kv0 + c;
        // a key row past N (zero-filled by the copy) must give P = 0: its
        // score 0 is not covered by L, and exp(0 - L) can overflow
        const bool kv_oob = kv >= N;
        bool ok = true;
        for (int it = 0; it < n_it; ++it) {
            const int st = it % QS;
            // every lane waits, then the warp votes: the tcgen05.ld/st below
            // are warp-collective and need all 32 lanes
            const bool w1 = mbar_wait(s_full, it & 1, abort_flag, p.status, 26);
            const bool w2 = w1 && mbar_wait(&qd_full[st], (it / QS) & 1, abort_flag, p.status, 27);
            if (!__all_sync(0xffffffffu, w2)) { ok = false; break; }
            tc_fence_after();
            const int q_base = (i_start + it % n_i) * kBQ;
            const bool diag = p.causal && (q_base + q0w < kv0 + kBKV);
            // some query of this slice is W or more rows below some key of the tile
            const bool wmask = win > 0 && (q_base + q0w + 16 * kNCH - 1 - kv0 >= win);
            const float *ldst = ld_smem + st * 2 * kBQ;  // -L log2(e) [128], then D [128]
            // ---- phase 1: P^T (16-bit pairs), kept in registers for phase 2
            uint32_t pp[kNCH][8];
            uint32_t sv[32];  // S^T of two chunks at a time
#pragma unroll
            for (int ch = 0; ch < kNCH; ++ch) {
                const int qc = q0w + ch * 16;  // first query column of this chunk
                const int q_first = q_base + qc;
                if ((ch & 1) == 0) {
                    tmem_ld_x32(lane_base + kColS + qc, sv);
                    tmem_ld_wait_x32(sv);
                }
                const uint32_t *s = sv + 16 * (ch & 1);
                // the chunk's 16 values of -L log2(e) in four 16-byte loads
                float nl[16];
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const float4 f = *reinterpret_cast<const float4 *>(ldst + qc + 4 * k);
                    nl[4 * k] = f.x;
                    nl[4 * k + 1] = f.y;
                    nl[4 * k + 2] = f.z;
                    nl[4 * k + 3] = f.w;
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
                    if (wmask) {  // sliding window: visible iff q - kv < W
                        if (q_first + r - kv >= win) p0 = 0.0f;
                        if (q_first + r + 1 - kv >= win) p1 = 0.0f;
                    }
                    pp[ch][r / 2] = BF16 ? pack_bf16x2(p0, p1) : pack_f16x2(p0, p1);
                }
                if (kv_oob) {  // P = 0, hence dS = 0, for the whole row
#pragma unroll
                    for (int r = 0; r < 8; ++r) pp[ch][r] = 0u;
                }
                __syncwarp();
                // P^T of this chunk goes into the first 8 of the chunk's own S^T
                // columns [qc, qc + 16), which this warp has read and no other reads
                tmem_st_x8(lane_base + kColS + qc, pp[ch]);
            }
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(p_ready);
            // ---- phase 2: dS^T = P^T o (dP^T - D), from the rounded P^T above
            const bool w3 = mbar_wait(dp_full, it & 1, abort_flag, p.status, 31);
            if (!__all_sync(0xffffffffu, w3)) { ok = false; break; }
            tc_fence_after();
            uint8_t *ds_row = smem + L::OFF_DS + hf * L::DS_BOX + c * 128;
            // dP^T one chunk at a time, each chunk's load issued before the
            // previous chunk's arithmetic (the wait then finds it done)
            uint32_t dpv[2][16];
            uint32_t ddk[kNCH][8];  // packed dS^T, kept for the shared-memory copy
            tmem_ld_x16(lane_base + kColDP + q0w, dpv[0]);
#pragma unroll
            for (int ch = 0; ch < kNCH; ++ch) {
                const int qc = q0w + ch * 16;
                tmem_ld_wait_x16(dpv[ch & 1]);  // the only load outstanding
                if (ch + 1 < kNCH) tmem_ld_x16(lane_base + kColDP + qc + 16, dpv[(ch + 1) & 1]);
                const uint32_t *dp = dpv[ch & 1];
                float dv_[16];  // the chunk's 16 values of D
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const float4 f = *reinterpret_cast<const float4 *>(ldst + kBQ + qc + 4 * k);
                    dv_[4 * k] = f.x;
                    dv_[4 * k + 1] = f.y;
                    dv_[4 * k + 2] = f.z;
                    dv_[4 * k + 3] = f.w;
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
                // dS^T into the last 8 of the chunk's 16 S^T columns
                tmem_st_x8(lane_base + kColS + qc + 8, dd);
                if (DQ && ch == kNCH / 2 - 1) {
                    // the first half of this warp's chunks is in tensor memory:
                    // the dK MMAs for those queries may start
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
            if constexpr (DQ) {
                // the shared-memory copy for dQ^T after ds_ready, so that dK and
                // the next S^T do not wait for these stores; dQ^T waits on ds_smem
#pragma unroll
                for (int ch = 0; ch < kNCH; ++ch)
#pragma unroll
                    for (int q = 0; q < 2; ++q)
                        *reinterpret_cast<uint4 *>(ds_row + (((2 * ch + q) ^ (c & 7)) << 4)) =
                            make_uint4(ddk[ch][4 * q], ddk[ch][4 * q + 1], ddk[ch][4 * q + 2], ddk[ch][4 * q + 3]);
                fence_proxy_async_smem();
                mbar_arrive(ds_smem);
            }
        }
        // ------------------------------- epilogue: dV (warps 0-3), dK (warps 4-7)
        bool ok2 = ok && warp < 8 && mbar_wait(acc_done, 0, abort_flag, p.status, 28);
        __syncwarp();
        if (warp < 8) ok2 = named_bar_and(1 + hf, 128, ok2);  // uniform per warp group
        if (ok2) {
            tc_fence_after();
            // the first Q/dO stage is idle after the last MMA: dV goes to its Q
            // buffer, dK to its dO buffer
            uint8_t *stage = hf == 0 ? q_stage(0) : do_stage(0);
            const uint32_t col = hf == 0 ? kColDV : kColDK;
            const float f = hf == 0 ? 1.0f : p.scale;
#pragma unroll 1
            for (int c0 = 0; c0 < D; c0 += 32) {
                uint32_t o[32];
                tmem_ld_x32(lane_base + col + c0, o);
                tmem_ld_wait_x32(o);
                uint32_t w[16];
#pragma unroll
                for (int x = 0; x < 16; ++x) {
                    const float a0 = __uint_as_float(o[2 * x]) * f;
                    const float a1 = __uint_as_float(o[2 * x + 1]) * f;
                    w[x] = BF16 ? pack_bf16x2(a0, a1) : pack_f16x2(a0, a1);
                }
                if (packed) {
                    // packed rows: a 128-row box past this sequence's end would
                    // overwrite the next sequence, so each thread stores its row
                    if (kv < N) {
                        uint4 *dst = reinterpret_cast<uint4 *>(static_cast<uint8_t *>(hf == 0 ? p.dv : p.dk) +
                                                               ((size_t)(row0 + kv) * p.Hkv + g) * (D * 2));
#pragma unroll
                        for (int q = 0; q < 4; ++q)
                            dst[c0 / 8 + q] = make_uint4(w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]);
                    }
                } else {
                    uint8_t *rowp = stage + (c0 >> 6) * L::BOX_KV + c * 128;
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const int chunk = ((c0 & 63) >> 3) + q;
                        *reinterpret_cast<uint4 *>(rowp + ((chunk ^ (c & 7)) << 4)) =
                            make_uint4(w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]);
                    }
                }
            }
            if (!packed) {
                fence_proxy_async_smem();
                named_bar_sync(1 + hf, 128);
                if (c == 0) {
                    const CUtensorMap *tm = hf == 0 ? &tm_dv : &tm_dk;
                    for (int bx = 0; bx < L::NBOX; ++bx) tma_store_3d(tm, stage + bx * L::BOX_KV, bx * 64, kv0, bg);
                    bulk_commit();
                    bulk_wait_read_all();
                }
            }
        }
        __syncwarp();
    } else {
        // ------------------- warps 8-15: dQ^T read-out and atomic reduction
        // Warp w reads TMEM lane quarter w % 4 (lane = head-dim index t) and
        // query columns 64 hf .. + 63 (hf = (w - 8) / 4).
        const int hf = (warp - 8) >> 2;
        const int quarter = warp & 3;
        const int t = quarter * 32 + lane;
        const uint32_t lane_base = tmem + ((uint32_t)(quarter * 32) << 16);
        for (int it = 0; DQ && it < n_it; ++it) {
            const bool got = mbar_wait(dq_full, it & 1, abort_flag, p.status, 29);
            if (!__all_sync(0xffffffffu, got)) break;
            tc_fence_after();
            uint32_t v[64];
            tmem_ld_x32(lane_base + kColDQ + hf * 64, v);
            tmem_ld_x32(lane_base + kColDQ + hf * 64 + 32, v + 32);
            tmem_ld_wait_x32(v);
            tmem_ld_wait_x32(v + 32);
            tc_fence_before();
            mbar_arrive(dq_free);
            const int h = g * G + it / n_i;
            const int q_first = (i_start + it % n_i) * kBQ + hf * 64;
            const int rows = min(64, N - q_first);
            if (t < D) {
                // element (q, t) of this head's dQ: consecutive lanes touch
                // consecutive floats (one 128-byte line per warp and row)
                if (packed) {  // packed: [total][Hq][d]
                    float *dst = p.dq_acc + ((size_t)(row0 + q_first) * p.Hq + h) * D + t;
                    const size_t rstride = (size_t)p.Hq * D;
#pragma unroll
                    for (int r = 0; r < 64; ++r)
                        if (r < rows) atomicAdd(dst + (size_t)r * rstride, __uint_as_float(v[r]));
                } else {  // dense: [B][Hq][N][d], constant row stride
                    float *dst = p.dq_acc + ((size_t)(b * p.Hq + h) * N + q_first) * D + t;
#pragma unroll
                    for (int r = 0; r < 64; ++r)
                        if (r < rows) atomicAdd(dst + (size_t)r * D, __uint_as_float(v[r]));
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

// D[row] = sum_c dO[row, c] * O[row, c]; also zeroes the fp32 dQ accumulator.
// 16 lanes per row, 16-byte loads.  Rows are taken in memory order; in the
// packed layout row t * Hq + h is stored at D[h * total + t] (the LSE layout).
template <bool BF16>
__global__ void __launch_bounds__(256) bwd_pre_kernel(const uint4 *__restrict__ o, const uint4 *__restrict__ dO,
                                                      float *__restrict__ Dvec, float4 *__restrict__ dq_acc,
                                                      long rows, int d, long acc_vec4, int Hq, long total,
                                                      int varlen) {
    const long tid = (long)blockIdx.x * blockDim.x + threadIdx.x;
    const long nthreads = (long)gridDim.x * blockDim.x;
    const int vec_per_row = d / 8;  // 8 elements per uint4
    // each warp takes two rows per trip (16 lanes each); the trip count is
    // uniform across the warp so the full-mask shuffles below are convergent
    const long warp_id = tid >> 5;
    const long nwarps = nthreads >> 5;
    const int half = (threadIdx.x >> 4) & 1;
    const int sub = threadIdx.x & 15;
    for (long base = warp_id * 2; base < rows; base += nwarps * 2) {
        const long row = base + half;
        float acc = 0.0f;
        if (row < rows) {
            for (int v = sub; v < vec_per_row; v += 16) {
                const uint4 a = o[row * vec_per_row + v];
                const uint4 bv = dO[row * vec_per_row + v];
                const uint32_t aw[4] = {a.x, a.y, a.z, a.w};
                const uint32_t bw[4] = {bv.x, bv.y, bv.z, bv.w};
#pragma unroll
                for (int x = 0; x < 4; ++x) {
                    const float2 af = unpack2<BF16>(aw[x]);
                    const float2 bf = unpack2<BF16>(bw[x]);
                    acc = fmaf(af.x, bf.x, acc);
                    acc = fmaf(af.y, bf.y, acc);
                }
            }
        }
#pragma unroll
        for (int off = 8; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
        if (sub == 0 && row < rows) Dvec[varlen ? (row % Hq) * total + row / Hq : row] = acc;
    }
    const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
    for (long i = tid; i < acc_vec4; i += nthreads) dq_acc[i] = z;
}

// dQ = scale * dQacc in the element type; 8 elements per thread.
template <bool BF16>
__global__ void __launch_bounds__(256) bwd_dq_kernel(const float4 *__restrict__ acc, uint4 *__restrict__ dq,
                                                     long n8, float scale) {
    const long nthreads = (long)gridDim.x * blockDim.x;
    for (long i = (long)blockIdx.x * blockDim.x + threadIdx.x; i < n8; i += nthreads) {
        const float4 a = acc[2 * i];
        const float4 c = acc[2 * i + 1];
        uint4 out;
        if constexpr (BF16) {
            out = make_uint4(pack_bf16x2(a.x * scale, a.y * scale), pack_bf16x2(a.z * scale, a.w * scale),
                             pack_bf16x2(c.x * scale, c.y * scale), pack_bf16x2(c.z * scale, c.w * scale));
        } else {
            out = make_uint4(pack_f16x2(a.x * scale, a.y * scale), pack_f16x2(a.z * scale, a.w * scale),
                             pack_f16x2(c.x * scale, c.y * scale), pack_f16x2(c.z * scale, c.w * scale));
        }
        dq[i] = out;
    }
}

// ---------------------------------------------------------------------------
// Second pass of the deterministic backward ([V2] section 7.2: dQ either by
// atomic addition, as above, or by a separate pass).  The first pass is
// bwd_main_kernel<D, BF16, false>, which produces dK and dV only.  Here every
// CTA owns one 128-row Q tile of one query head and walks the K/V tiles of its
// key/value head in order, so each element of dQ is accumulated by the tensor
// core in a fixed order and stored once: the result does not depend on
// scheduling.  Per K/V tile j, from the stored L and D:
//   S = Q K_j^T, dP = dO V_j^T              (both operands in shared memory)
//   P = exp2(S scale log2(e) - L log2(e)), dS = P o (dP - D)
//   dQ += dS K_j                             (A = dS from tensor memory)
// Tensor memory, lane = query row:
//   [0, 128), [128, 256)  S of even / odd tiles; dS (16-bit pairs) is written
//                          over the S columns its own warp has already read
//   [256, 384)            dP
//   [384, 384 + d)        dQ
// Warps: 0-7 dS (warp w: lane quarter w % 4, keys 64 (w / 4) .. + 63), then
// the dQ epilogue; 8 TMA producer; 9 MMA issuer + tensor-memory owner.
constexpr int kDqThreads = 320;
constexpr int kDqSoftmaxThreads = 256;
constexpr int kDqProducerWarp = 8, kDqMmaWarp = 9;
constexpr uint32_t kDqColS = 0, kDqColDP = 256, kDqColDQ = 384;

template <int D>
struct DqLayout {
    static constexpr int NBOX = D / 64;
    static constexpr int TILE = 128 * D * 2;  // one 128-row tile of Q, dO, K or V
    static constexpr int BOX = 128 * 128;     // one 64-column box of a tile
    static constexpr int KS = D == 128 ? 3 : 4;  // K is held until dQ of its tile
    static constexpr int VS = D == 128 ? 2 : 4;  // V only until dP of its tile
    static constexpr int OFF_Q = 0;
    static constexpr int OFF_DO = OFF_Q + TILE;
    static constexpr int OFF_K = OFF_DO + TILE;
    static constexpr int OFF_V = OFF_K + KS * TILE;
    static constexpr int OFF_BAR = OFF_V + VS * TILE;
    // q_full, k_full[KS], k_empty[KS], v_full[VS], v_empty[VS], sdp_full[2],
    // ds_ready[2], dp_free, acc_done, drain
    static constexpr int NBAR = 1 + 2 * KS + 2 * VS + 4 + 3;
    static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
    static constexpr int BYTES = OFF_MISC + 16;
    static constexpr int SLACK = 512;
    static constexpr int ALLOC = BYTES + SLACK;
    static_assert(ALLOC <= 227 * 1024, "shared memory");
};

struct DqParams {
    const float *lse;
    const float *Dvec;
    void *dq;                // packed layout: stored row by row
    unsigned int *status;
    const int *cu_seqlens;   // packed layout: sequence b is rows cu[b] .. cu[b+1]-1
    int varlen, total;
    int Hq, Hkv, N, nq, nkv;
    int causal;
    int window;  // > 0: query r sees keys r - window + 1 .. r only
    int group;   // query planes per CTA-order group (grid_order.cuh)
    float scale, scale_log2;
};

template <int D, bool BF16, bool GENERAL>
__global__ void __launch_bounds__(kDqThreads, 1)
    bwd_dq_pass_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                       const __grid_constant__ CUtensorMap tm_dq, const DqParams p) {
    using L = DqLayout<D>;
    constexpr int KS = L::KS, VS = L::VS;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t pad = (1024u - (smem_u32(smem_raw) & 1023u)) & 1023u;
    if (pad > (uint32_t)L::SLACK) {  // uniform across the CTA; nothing started yet
        if (threadIdx.x == 0) record_bad_launch(p.status);
        return;
    }
    uint8_t *smem = smem_raw + pad;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::OFF_BAR);
    uint64_t *q_full = bars;
    uint64_t *k_full = q_full + 1;
    uint64_t *k_empty = k_full + KS;
    uint64_t *v_full = k_empty + KS;
    uint64_t *v_empty = v_full + VS;
    uint64_t *sdp_full = v_empty + VS;
    uint64_t *ds_ready = sdp_full + 2;
    uint64_t *dp_free = ds_ready + 2;
    uint64_t *acc_done = dp_free + 1;
    uint64_t *drain = acc_done + 1;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L::OFF_MISC);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::OFF_MISC + 4);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int win = GENERAL ? p.window : 0;
    const bool packed = GENERAL && p.varlen;

    // CTA order: query planes in L2-sized groups, longest causal tiles first
    int bh, qt_lin;
    grid_decode(blockIdx.x, (int)(gridDim.x / p.nq), p.nq, p.group, bh, qt_lin);
    const int qt = p.causal ? (p.nq - 1 - qt_lin) : qt_lin;
    const int b = bh / p.Hq;
    const int h = bh - b * p.Hq;
    const int hk = h / (p.Hq / p.Hkv);
    const int kv_plane = b * p.Hkv + hk;
    const int q0 = qt * 128;
    // rows of this sequence (packed layout: rows row0 .. row0 + N - 1)
    int N = p.N, row0 = 0;
    if (packed) {
        row0 = p.cu_seqlens[b];
        N = p.cu_seqlens[b + 1] - row0;
        if (N < 0 || N > p.N || row0 < 0 || row0 + N > p.total) {
            if (threadIdx.x == 0 && qt_lin == 0) record_bad_args(p.status);
            return;  // uniform across the CTA, nothing started yet
        }
    }
    if (q0 >= N) return;  // Q tile past the end of a shorter sequence
    const int nkv = (N + 127) / 128;
    const int j_end = p.causal ? min(qt + 1, nkv) : nkv;
    // sliding window of W keys: the first key any row of this tile sees is
    // q0 - W + 1, so K/V tiles before its tile are skipped
    const int j_lo = win > 0 ? max(0, q0 - win + 1) / 128 : 0;
    const int n_j = j_end - j_lo;  // K/V tiles j_lo .. j_end - 1, counted from 0 below

    if (threadIdx.x == 0) {
        mbar_init(q_full, 1);
        for (int s = 0; s < KS; ++s) { mbar_init(&k_full[s], 1); mbar_init(&k_empty[s], 1); }
        for (int s = 0; s < VS; ++s) { mbar_init(&v_full[s], 1); mbar_init(&v_empty[s], 1); }
        for (int s = 0; s < 2; ++s) { mbar_init(&sdp_full[s], 1); mbar_init(&ds_ready[s], kDqSoftmaxThreads); }
        mbar_init(dp_free, kDqSoftmaxThreads);
        mbar_init(acc_done, 1);
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == kDqMmaWarp) {
        tmem_alloc(tmem_slot, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == kDqProducerWarp) {
        // ------------------------------------------------------ TMA producer
        if (lane == 0) {
            prefetch_tmap(&tm_k);
            prefetch_tmap(&tm_v);
            mbar_arrive_expect_tx(q_full, 2 * L::TILE);
            for (int bx = 0; bx < L::NBOX; ++bx) {
                const int c1 = packed ? h : q0, c2 = packed ? row0 + q0 : bh;
                tma_load_3d(smem + L::OFF_Q + bx * L::BOX, &tm_q, q_full, bx * 64, c1, c2);
                tma_load_3d(smem + L::OFF_DO + bx * L::BOX, &tm_do, q_full, bx * 64, c1, c2);
            }
            int nk = 0, nv = 0;  // tiles whose copies were issued
            for (int j = 0; j < n_j; ++j) {
                const int ks = j % KS;
                if (j >= KS && !mbar_wait(&k_empty[ks], ((j / KS) + 1) & 1, abort_flag, p.status, 41)) break;
                mbar_arrive_expect_tx(&k_full[ks], L::TILE);
                for (int bx = 0; bx < L::NBOX; ++bx)
                    tma_load_3d(smem + L::OFF_K + ks * L::TILE + bx * L::BOX, &tm_k, &k_full[ks], bx * 64,
                                packed ? hk : (j_lo + j) * 128, packed ? row0 + (j_lo + j) * 128 : kv_plane);
                ++nk;
                const int vs = j % VS;
                if (j >= VS && !mbar_wait(&v_empty[vs], ((j / VS) + 1) & 1, abort_flag, p.status, 42)) break;
                mbar_arrive_expect_tx(&v_full[vs], L::TILE);
                for (int bx = 0; bx < L::NBOX; ++bx)
                    tma_load_3d(smem + L::OFF_V + vs * L::TILE + bx * L::BOX, &tm_v, &v_full[vs], bx * 64,
                                packed ? hk : (j_lo + j) * 128, packed ? row0 + (j_lo + j) * 128 : kv_plane);
                ++nv;
            }
            if (*abort_flag) {
                // let copies already in flight land before the CTA exits
                mbar_wait_drain(q_full, 0, 10000000ull);
                for (int t = max(0, nk - KS); t < nk; ++t)
                    mbar_wait_drain(&k_full[t % KS], (t / KS) & 1, 10000000ull);
                for (int t = max(0, nv - VS); t < nv; ++t)
                    mbar_wait_drain(&v_full[t % VS], (t / VS) & 1, 10000000ull);
            }
        }
        __syncwarp();
    } else if (warp == kDqMmaWarp) {
        // ------------------------------------------------------- MMA issuer
        if (lane == 0) {
            constexpr uint32_t fmt = BF16 ? 1u : 0u;
            constexpr uint32_t idesc_sdp = make_idesc(128, 128, fmt, false, false);  // K-major both
            constexpr uint32_t idesc_dq = make_idesc(128, D, fmt, false, true);      // A tmem, B MN-major
            const uint64_t q_desc = make_sdesc_sw128(smem_u32(smem + L::OFF_Q), 16, 1024);
            const uint64_t do_desc = make_sdesc_sw128(smem_u32(smem + L::OFF_DO), 16, 1024);
            const uint64_t k_desc0 = make_sdesc_sw128(smem_u32(smem + L::OFF_K), 16, 1024);
            // K as the MN-major B of dQ += dS K (N = head dim, contiguous)
            const uint64_t km_desc0 = make_sdesc_sw128(smem_u32(smem + L::OFF_K), L::BOX, 1024);
            const uint64_t v_desc0 = make_sdesc_sw128(smem_u32(smem + L::OFF_V), 16, 1024);

            // dQ += dS_t K_t; 16 keys = 8 packed columns of A, 16 rows (2048
            // bytes) of B per step.  Keys 64 h + 16 m .. + 15 of the tile have
            // their dS at columns 64 h + 8 m .. + 7 of the S buffer.
            auto issue_dq = [&](int t) -> bool {
                const int sb = t & 1;
                if (!mbar_wait(&ds_ready[sb], (t >> 1) & 1, abort_flag, p.status, 43)) return false;
                tc_fence_after();
                const int ks = t % KS;
                const uint64_t km_desc = sdesc_advance(km_desc0, ks * L::TILE);
                const uint32_t a_col = tmem + kDqColS + sb * 128;
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)
                    mma_f16_ts(tmem + kDqColDQ, a_col + (kk >> 2) * 64 + (kk & 3) * 8,
                               sdesc_advance(km_desc, kk * 2048), idesc_dq, (t > 0 || kk > 0) ? 1u : 0u);
                mma_commit(&k_empty[ks]);
                return true;
            };

            bool ok = mbar_wait(q_full, 0, abort_flag, p.status, 44);
            for (int j = 0; ok && j < n_j; ++j) {
                const int ks = j % KS, vs = j % VS, sb = j & 1;
                if (!mbar_wait(&k_full[ks], (j / KS) & 1, abort_flag, p.status, 45)) { ok = false; break; }
                tc_fence_after();
                // S_j into buffer sb: its previous contents, dS_{j-2}, were read
                // by the dQ MMAs issued before (the MMAs run in issue order)
                const uint64_t k_desc = sdesc_advance(k_desc0, ks * L::TILE);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t off = (kk >> 2) * L::BOX + (kk & 3) * 32;
                    mma_f16_ss(tmem + kDqColS + sb * 128, sdesc_advance(q_desc, off), sdesc_advance(k_desc, off),
                               idesc_sdp, kk > 0 ? 1u : 0u);
                }
                // dP_j: the dS warps have loaded dP_{j-1} into registers
                if (j > 0 && !mbar_wait(dp_free, (j - 1) & 1, abort_flag, p.status, 46)) { ok = false; break; }
                if (!mbar_wait(&v_full[vs], (j / VS) & 1, abort_flag, p.status, 47)) { ok = false; break; }
                tc_fence_after();
                const uint64_t v_desc = sdesc_advance(v_desc0, vs * L::TILE);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t off = (kk >> 2) * L::BOX + (kk & 3) * 32;
                    mma_f16_ss(tmem + kDqColDP, sdesc_advance(do_desc, off), sdesc_advance(v_desc, off), idesc_sdp,
                               kk > 0 ? 1u : 0u);
                }
                mma_commit(&v_empty[vs]);
                mma_commit(&sdp_full[sb]);
                // dQ of the previous tile runs while the dS warps work on this one
                if (j > 0 && !issue_dq(j - 1)) { ok = false; break; }
            }
            if (ok && n_j > 0) ok = issue_dq(n_j - 1);
            if (ok) mma_commit(acc_done);
            // every MMA issued above has completed once `drain` flips
            mma_commit(drain);
            mbar_wait_drain(drain, 0, 100000000ull);
        }
        __syncwarp();
    } else {
        // ------------------------------------------- warps 0-7: dS, epilogue
        const int hf = warp >> 2;
        const int quarter = warp & 3;
        const int r = quarter * 32 + lane;  // query row == TMEM lane
        const uint32_t lane_base = tmem + ((uint32_t)(quarter * 32) << 16);
        const int q = q0 + r;
        const bool q_in = q < N;
        const size_t li = packed ? (size_t)h * p.total + row0 + q : (size_t)bh * N + q;
        // rows past N: P = 0 (their dQ rows are not stored)
        const float nl2 = q_in ? -p.lse[li] * 1.4426950408889634f : -INFINITY;
        const float dq_d = q_in ? p.Dvec[li] : 0.0f;
        // keys this row attends to: kv_lo .. kv_last (causal: up to q; never
        // a key past N; sliding window: from q - W + 1)
        const int kv_last = p.causal ? min(q, N - 1) : N - 1;
        const int kv_lo = win > 0 ? q - win + 1 : 0;
        const float2 sl2 = make_float2(p.scale_log2, p.scale_log2);
        const float2 nl2x2 = make_float2(nl2, nl2);
        const float2 dx2 = make_float2(dq_d, dq_d);
        bool ok = true;
        for (int j = 0; j < n_j; ++j) {
            const int sb = j & 1;
            const bool got = mbar_wait(&sdp_full[sb], (j >> 1) & 1, abort_flag, p.status, 48);
            if (!__all_sync(0xffffffffu, got)) { ok = false; break; }
            tc_fence_after();
            uint32_t dp[64];
            tmem_ld_x32(lane_base + kDqColDP + hf * 64, dp);
            tmem_ld_x32(lane_base + kDqColDP + hf * 64 + 32, dp + 32);
            tmem_ld_wait_x32(dp);
            tmem_ld_wait_x32(dp + 32);
            tc_fence_before();
            mbar_arrive(dp_free);
            const int kv_first = (j_lo + j) * 128 + hf * 64;
            const bool masked = kv_first + 63 > kv_last || kv_first < kv_lo;
            const uint32_t s_cols = lane_base + kDqColS + sb * 128 + hf * 64;
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                uint32_t s[32];
                tmem_ld_x32(s_cols + 32 * c, s);
                tmem_ld_wait_x32(s);
                uint32_t dd[16];
#pragma unroll
                for (int x = 0; x < 32; x += 2) {
                    const float2 t = ffma2(make_float2(__uint_as_float(s[x]), __uint_as_float(s[x + 1])), sl2, nl2x2);
                    float p0 = ex2_approx(t.x);
                    float p1 = ex2_approx(t.y);
                    if (masked) {
                        const int kv = kv_first + 32 * c + x;
                        if (kv > kv_last || kv < kv_lo) p0 = 0.0f;
                        if (kv + 1 > kv_last || kv + 1 < kv_lo) p1 = 0.0f;
                    }
                    // P rounded to the element type, as in the K/V-tile pass (where
                    // the same rounded P feeds dV), so both passes use one dS
                    const float2 pr = unpack2<BF16>(BF16 ? pack_bf16x2(p0, p1) : pack_f16x2(p0, p1));
                    const float2 ds = fmul2(pr,
                                            fsub2(make_float2(__uint_as_float(dp[32 * c + x]),
                                                              __uint_as_float(dp[32 * c + x + 1])),
                                                  dx2));
                    dd[x / 2] = BF16 ? pack_bf16x2(ds.x, ds.y) : pack_f16x2(ds.x, ds.y);
                }
                __syncwarp();
                // keys 32 c .. 32 c + 31 of this half -> packed columns 16 c .. + 15,
                // all already read by this thread (own lane, columns < 32 (c + 1))
                tmem_st_x16(s_cols + 16 * c, dd);
            }
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(&ds_ready[sb]);
        }
        // ------------------------------------------------ epilogue: dQ store
        bool ok2 = ok && mbar_wait(acc_done, 0, abort_flag, p.status, 49);
        __syncwarp();
        ok2 = named_bar_and(1, kDqSoftmaxThreads, ok2);
        if (ok2) {
            tc_fence_after();
            // Q is no longer read once every MMA has completed: its buffer
            // stages the output tile
            uint8_t *stage = smem + L::OFF_Q;
#pragma unroll 1
            for (int c0 = hf * (D / 2); c0 < (hf + 1) * (D / 2); c0 += 32) {
                uint32_t o[32];
                tmem_ld_x32(lane_base + kDqColDQ + c0, o);
                tmem_ld_wait_x32(o);
                uint32_t w[16];
#pragma unroll
                for (int x = 0; x < 16; ++x) {
                    const float a0 = __uint_as_float(o[2 * x]) * p.scale;
                    const float a1 = __uint_as_float(o[2 * x + 1]) * p.scale;
                    w[x] = BF16 ? pack_bf16x2(a0, a1) : pack_f16x2(a0, a1);
                }
                if (packed) {
                    // packed rows: each thread stores its own row (a 128-row box
                    // past this sequence's end would overwrite the next one)
                    if (q_in) {
                        uint4 *dst = reinterpret_cast<uint4 *>(static_cast<uint8_t *>(p.dq) +
                                                               ((size_t)(row0 + q) * p.Hq + h) * (D * 2));
#pragma unroll
                        for (int x = 0; x < 4; ++x)
                            dst[c0 / 8 + x] = make_uint4(w[4 * x], w[4 * x + 1], w[4 * x + 2], w[4 * x + 3]);
                    }
                } else {
                    uint8_t *rowp = stage + (c0 >> 6) * L::BOX + r * 128;
#pragma unroll
                    for (int x = 0; x < 4; ++x) {
                        const int chunk = ((c0 & 63) >> 3) + x;
                        *reinterpret_cast<uint4 *>(rowp + ((chunk ^ (r & 7)) << 4)) =
                            make_uint4(w[4 * x], w[4 * x + 1], w[4 * x + 2], w[4 * x + 3]);
                    }
                }
            }
            if (!packed) {
                fence_proxy_async_smem();
                named_bar_sync(1, kDqSoftmaxThreads);
                if (threadIdx.x == 0) {
                    for (int bx = 0; bx < L::NBOX; ++bx)
                        tma_store_3d(&tm_dq, stage + bx * L::BOX, bx * 64, q0, bh);
                    bulk_commit();
                    bulk_wait_read_all();
                }
            }
        }
        __syncwarp();
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kDqMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// Longest sequence fa_bwd runs with the persistent main kernel.  Measured
// on a GB300 against one CTA per work item (bf16, d = 128, 16 heads, causal):
// N = 512 1.09x, N = 1024 1.04x, N = 2048 0.99-1.00x.
constexpr int kPersistBwdMaxN = 1024;

int elementwise_blocks() {
    int dev = 0, sms = 152;
    if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    return sms * 8;
}

// two_pass = false: pre, main (with dQ atomics), dQ conversion.
// two_pass = true:  pre (D only), main without dQ, bwd_dq_pass_kernel.
template <int D, bool BF16>
cudaError_t launch_bwd_t(const BwdArgs &a, cudaStream_t st, bool two_pass) {
    using L = BwdLayout<D>;
    const CUtensorMapDataType dt = BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    const SeqLayout &lay = a.lay;
    CUtensorMap tq, tk, tv, tdo, tdk, tdv, tdq;
    if (!make_tmap_tiles(&tq, a.q, dt, D, lay, a.Hq, kBQ) || !make_tmap_tiles(&tdo, a.dO, dt, D, lay, a.Hq, kBQ) ||
        !make_tmap_tiles(&tk, a.k, dt, D, lay, a.Hkv, kBKV) || !make_tmap_tiles(&tv, a.v, dt, D, lay, a.Hkv, kBKV) ||
        !make_tmap_tiles(&tdk, a.dk, dt, D, lay, a.Hkv, kBKV) ||
        !make_tmap_tiles(&tdv, a.dv, dt, D, lay, a.Hkv, kBKV) ||
        (two_pass && !make_tmap_tiles(&tdq, a.dq, dt, D, lay, a.Hq, kBQ)))
        return cudaErrorInvalidValue;

    const long rows = (long)lay.total * a.Hq;  // dense: total = B * N
    const int eb = elementwise_blocks();
    bwd_pre_kernel<BF16><<<eb, 256, 0, st>>>(static_cast<const uint4 *>(a.o), static_cast<const uint4 *>(a.dO),
                                             a.D, reinterpret_cast<float4 *>(a.dq_acc), rows, D,
                                             two_pass ? 0 : rows * D / 4, a.Hq, (long)lay.total, lay.varlen);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;

    const bool general = a.window > 0 || lay.varlen;
    auto main_kernel = two_pass ? (general ? bwd_main_kernel<D, BF16, false, true> : bwd_main_kernel<D, BF16, false, false>)
                                : (general ? bwd_main_kernel<D, BF16, true, true> : bwd_main_kernel<D, BF16, true, false>);
    e = cudaFuncSetAttribute(main_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, L::ALLOC);
    if (e != cudaSuccess) return e;
    BwdParams p;
    p.lse = a.lse;
    p.Dvec = a.D;
    p.dq_acc = a.dq_acc;
    p.dk = a.dk;
    p.dv = a.dv;
    p.status = device_status_ptr();
    p.cu_seqlens = lay.cu_seqlens;
    p.varlen = lay.varlen;
    p.total = lay.total;
    p.Hq = a.Hq;
    p.Hkv = a.Hkv;
    p.N = a.N;
    p.nkv = (a.N + kBKV - 1) / kBKV;
    p.nq = (a.N + kBQ - 1) / kBQ;
    p.causal = a.causal;
    p.window = a.window;
    p.scale = a.scale;
    p.scale_log2 = a.scale * 1.4426950408889634f;
    int sms = 0;
    {
        int dev = 0;
        if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
        if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    }
    p.group = grid_group_planes(a.B * a.Hkv, p.nkv, sms);
    const long long grid = (long long)p.nkv * a.B * a.Hkv;
    // short sequences: the persistent main kernel (fa_bwd_persist.cu), same
    // arithmetic, work items handed out dynamically, per-item set-up and
    // epilogue overlapped (it stores dK/dV rows 32 bytes at a time)
    const bool aligned32 = ((reinterpret_cast<uintptr_t>(a.dk) | reinterpret_cast<uintptr_t>(a.dv)) & 31u) == 0;
    if (!two_pass && !general && aligned32 && a.N <= kPersistBwdMaxN) {
        e = launch_bwd_persist_main(a, st);
    } else {
        main_kernel<<<dim3((unsigned)grid), dim3(kThreads), L::ALLOC, st>>>(tq, tk, tv, tdo, tdk, tdv, p);
        e = cudaGetLastError();
    }
    if (e != cudaSuccess) return e;

    if (two_pass) {
        using LQ = DqLayout<D>;
        auto dq_kernel = general ? bwd_dq_pass_kernel<D, BF16, true> : bwd_dq_pass_kernel<D, BF16, false>;
        e = cudaFuncSetAttribute(dq_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, LQ::ALLOC);
        if (e != cudaSuccess) return e;
        DqParams pq2;
        pq2.lse = a.lse;
        pq2.Dvec = a.D;
        pq2.status = p.status;
        pq2.dq = a.dq;
        pq2.cu_seqlens = lay.cu_seqlens;
        pq2.varlen = lay.varlen;
        pq2.total = lay.total;
        pq2.Hq = a.Hq;
        pq2.Hkv = a.Hkv;
        pq2.N = a.N;
        pq2.nq = p.nq;
        pq2.nkv = p.nkv;
        pq2.causal = a.causal;
        pq2.window = a.window;
        pq2.scale = a.scale;
        pq2.scale_log2 = p.scale_log2;
        pq2.group = grid_group_planes(a.B * a.Hq, p.nq, sms);
        const long long grid2 = (long long)p.nq * a.B * a.Hq;
        dq_kernel<<<dim3((unsigned)grid2), dim3(kDqThreads), LQ::ALLOC, st>>>(tq, tk, tv, tdo, tdq, pq2);
        return cudaGetLastError();
    }

    bwd_dq_kernel<BF16><<<eb, 256, 0, st>>>(reinterpret_cast<const float4 *>(a.dq_acc),
                                            static_cast<uint4 *>(a.dq), rows * D / 8, a.scale);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd(const BwdArgs &a, cudaStream_t st, bool two_pass) {
    if (a.d == 128) return a.bf16 ? launch_bwd_t<128, true>(a, st, two_pass) : launch_bwd_t<128, false>(a, st, two_pass);
    if (a.d == 64) return a.bf16 ? launch_bwd_t<64, true>(a, st, two_pass) : launch_bwd_t<64, false>(a, st, two_pass);
    return cudaErrorInvalidValue;
}

}  // namespace fa
