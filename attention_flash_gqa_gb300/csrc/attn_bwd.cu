// Attention backward on tcgen05 tensor cores, for the forward in attn_fwd.cu. The main kernel here
// (a thread-block cluster per key tile) serves D = 512; D = 64, 128 and 256 use the cluster-free
// kernel in attn_bwd_small.cu. The prep and finalize kernels here serve every D. Given dO, lse and Delta = rowsum(dO * o):
//   P  = exp(scale * Q K^T - lse)        (recomputed; never stored)
//   dP = dO V^T,   dS = P * (dP - Delta)
//   dV = P^T dO,   dK = scale * dS^T Q,   dQ = scale * dS K
// Sources: "Root cause analysis: Gemma4 sliding-window BF16 cuDNN SDPA NaN on H100"
// ("Debug and validation results": the sliding-window backward must keep dQ/dK/dV
// finite in bf16 from finite dO) and the head_dim 512 path of "Gemma4 FFPA attention
// backend support ..." ("3x fwd / 6x bwd vs SDPA": the backward is where the time goes).
//
// Kernels:
//  1. bwd_prep: Delta per query row (fp32) and zeroing of the fp32 dQ accumulator.
//  2. bwd_main: one thread-block cluster per (KV tile of 128 keys, KV head); its
//     NC = D / 128 = 4 CTAs each own one 128-wide column slice c of D and accumulate dV_c
//     and dK_c for the tile in tensor memory while looping over every query head of the
//     GQA group and every query tile that can see the keys (causal / window tile
//     skipping), so dK and dV are summed over the group without atomics. A step is one
//     (head, query tile); steps are taken two at a time ("pair-steps").
//     The two full-width contractions are split across the cluster instead of being
//     recomputed per slice: CTAs 0, 1 ("S role") compute S = Q K^T, CTAs 2, 3 ("dP role")
//     dP = dO V^T, each for its own 64-query share of both steps of a pair-step at once:
//     one M = 128 product (rows = the two steps' shares, queries on TMEM lanes) over the
//     128 keys, so the full-width key (or value) tile streams once per two steps. An
//     S-role CTA turns its rows into P (bf16) and copies them into every CTA of the
//     cluster; its dP-role partner (same share) reads those rows, forms
//     dS = P (dP - Delta) and copies it likewise. Each CTA then runs its slice of the
//     three gradient products from the assembled per-step P / dS tiles [128 queries x 128
//     keys] in shared memory (P^T and dS^T read MN-major):
//       dV_c += P^T dO_c,   dK_c += dS^T Q_c,   dQ_c = dS K_c
//     dQ_c leaves tensor memory after every step and is added into an fp32 accumulator
//     with TMA bulk reduce-adds. Consumption of the exchanged tiles is signalled back to
//     their writers with multicast tcgen05.commit arrivals. P is double-buffered (one
//     buffer per step of a pair-step); dS is single-buffered.
//     Tensor memory (512 columns): [0,128) dV_c, [128,256) dK_c, [256,384) dQ_c,
//     [384,512) the role result of a pair-step.
//  3. bwd_finalize: dQ accumulator -> bf16.
#include <cuda_runtime.h>

#include <algorithm>
#include <type_traits>

#include "attn_internal.h"
#include "ptx.cuh"

namespace attn {
namespace {

constexpr int kB = 128;  // query tile = key tile = 128 rows
constexpr int kThreads = 192;
constexpr uint32_t kSlot = 16384;   // ring slot: one 128 x 64 bf16 sub-tile
constexpr uint32_t kSub = 16384;    // 128 rows x 128 bytes, 128-byte swizzle
constexpr uint32_t kSmemMax = 232448;

constexpr float kLog2e = 1.4426950408889634f;

// Configuration of the cluster kernel (D = 512: four CTAs, two per role).
template <int D>
struct Cfg {
    static constexpr int NC = D / 128;        // cluster size = slices of D
    static constexpr int NHALF = NC / 2;      // CTAs per role
    static constexpr int NQ = 128 / NHALF;    // queries of one role share per step
    static constexpr int NSUB = D / 64;       // 64-wide sub-tiles across D
    static constexpr uint32_t kPieceBytes = 128u * NQ * 2u;  // one role share of a step's P or dS
    static constexpr uint32_t kRemoteBytes = (NHALF - 1) * kPieceBytes;  // from the other writers
    static constexpr int kStages = 5;                                 // ring slots
    static constexpr uint32_t kOffP = 0;                              // P, two steps: [128 queries x 128 keys] bf16
    static constexpr uint32_t kOffDS = kOffP + 2 * 2 * kSub;          // dS, same layout
    static constexpr uint32_t kOffKc = kOffDS + 2 * kSub;             // K_c [128 keys x 128 dims], resident
    static constexpr uint32_t kOffStage = kOffKc + 2 * kSub;          // dQ staging (128 rows x 32 fp32)
    static constexpr uint32_t kOffRing = kOffStage + kSub;
    static constexpr uint32_t kOffBar = kOffRing + kStages * kSlot;
    static constexpr uint32_t kSmem = kOffBar + 512 + 1024;  // + slack for the 1024-byte alignment
    static_assert(kSmem <= kSmemMax, "shared memory budget");
    static_assert(NQ == 64, "the role split is written for D = 512");
};

struct BwdArgs {
    const float* lse;
    const float* delta;
    uint16_t *dK, *dV;
    const int32_t* cu_seqlens;
    unsigned* status;
    int Hq, Hkv, S, window, T;
    float scale, scale_log2;
};

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_main_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                    const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap tdo,
                    const __grid_constant__ CUtensorMap tqh, const __grid_constant__ CUtensorMap tdoh,
                    const __grid_constant__ CUtensorMap tdq, BwdArgs a) {
    using C = Cfg<D>;
    const uint32_t rank = cluster_ctarank();
    const int g = blockIdx.x / C::NC;  // KV head
    const bool s_role = rank < (uint32_t)C::NHALF;
    const int share = s_role ? (int)rank : (int)rank - C::NHALF;  // query share of the role work
    const int c0 = (int)rank * 128;  // this CTA's column slice of D
    const int seq = blockIdx.y;
    const int kv_tile = blockIdx.z;  // tile 0 sees the most queries: launched first
    int seq_start = 0, L = a.S, bcoord = seq;
    if (a.cu_seqlens) {
        seq_start = a.cu_seqlens[seq];
        L = a.cu_seqlens[seq + 1] - seq_start;
        bcoord = 0;
        // every CTA of the cluster reads the same slice and returns together, before any barrier
        if (!varlen_seq_ok(seq_start, L, a.T, a.S)) {
            if (threadIdx.x == 0 && blockIdx.x == 0 && kv_tile == 0) atomicOr(a.status, DEVSTAT_BOUNDS);
            return;
        }
    }
    const int k0 = kv_tile * kB;
    if (k0 >= L) return;  // the same for every CTA of the cluster
    const int G = a.Hq / a.Hkv;
    const int q_last = a.window > 0 ? min(L, k0 + kB - 1 + a.window) : L;  // exclusive bound on queries
    const int i_begin = k0 / kB, i_end = (q_last + kB - 1) / kB;
    const int n_qt = i_end - i_begin;
    const int n = G * n_qt;    // steps: (head, query tile)
    const int np = (n + 1) / 2;  // pair-steps: steps 2T and 2T + 1 (the latter absent when n is odd)

    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    const uint32_t sP = sbase + C::kOffP, sDS = sbase + C::kOffDS, sKc = sbase + C::kOffKc, sStage = sbase + C::kOffStage;
    const uint32_t sRing = sbase + C::kOffRing;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
    uint64_t* full = bars;
    uint64_t* empty = bars + C::kStages;
    uint64_t* r_full = bars + 2 * C::kStages;  // role result of a pair-step in TMEM complete
    uint64_t* r_free = r_full + 1;          // role result read out by the elementwise warps (128)
    uint64_t* p_full = r_free + 1;          // all of P(t) present in buffer t & 1 [2]
    uint64_t* ds_full = p_full + 2;         // all of dS(t) present
    uint64_t* p_free = ds_full + 1;         // (S role) every reader of this CTA's share of P in buffer b is done [2]
    uint64_t* ds_free = p_free + 2;         // (dP role) every reader of this CTA's share of dS is done
    uint64_t* dq_full = ds_free + 1;
    uint64_t* dq_free = dq_full + 1;
    uint64_t* kc_full = dq_free + 1;
    uint64_t* mma_idle = kc_full + 1;
    uint64_t* p_read = mma_idle + 1;  // (dP role) the elementwise warps have read P(t) [2]
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(p_read + 2);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (tid == 0) {
        for (int s = 0; s < C::kStages; ++s) {
            mbar_init(smem_u32(&full[s]), 1);
            mbar_init(smem_u32(&empty[s]), 1);
        }
        mbar_init(smem_u32(r_full), 1);
        mbar_init(smem_u32(r_free), 128);
        // exchange barriers: one arming arrive (with the bytes expected from other CTAs)
        // plus, for the share this CTA writes itself, the 64 threads that hold a step's rows
        for (int b = 0; b < 2; ++b) mbar_init(smem_u32(&p_full[b]), 1 + (s_role ? 64 : 0));
        mbar_init(smem_u32(ds_full), 1 + (s_role ? 0 : 64));
        // one multicast commit from every CTA's MMA (a dP-role CTA commits only after its
        // elementwise warps have also read P)
        for (int b = 0; b < 2; ++b) mbar_init(smem_u32(&p_free[b]), C::NC);
        mbar_init(smem_u32(ds_free), C::NC);
        mbar_init(smem_u32(dq_full), 1);
        mbar_init(smem_u32(dq_free), 128);
        mbar_init(smem_u32(kc_full), 1);
        mbar_init(smem_u32(mma_idle), 1);
        for (int b = 0; b < 2; ++b) mbar_init(smem_u32(&p_read[b]), 64);
        *abort_flag = 0;
        fence_mbar_init();
        // arm phase 0 of the exchange barriers (later phases are armed by the MMA issuer)
        for (int b = 0; b < 2; ++b)
            mbar_expect_tx(smem_u32(&p_full[b]), s_role ? C::kRemoteBytes : C::NHALF * C::kPieceBytes);
        mbar_expect_tx(smem_u32(ds_full), s_role ? C::NHALF * C::kPieceBytes : C::kRemoteBytes);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), 512);
        tmem_relinquish();
    }
    __syncthreads();
    cluster_sync_all();  // every CTA's barriers are initialised before any peer signals them
    tc_fence_after();
    const uint32_t tbase = *tmem_slot;
    const uint32_t tDV = tbase, tDK = tbase + 128, tDQ = tbase + 256, tR = tbase + 384;
    const int krow = seq_start + k0;
    const uint32_t p_rem = s_role ? C::kRemoteBytes : C::NHALF * C::kPieceBytes;
    const uint32_t ds_rem = s_role ? C::NHALF * C::kPieceBytes : C::kRemoteBytes;
    auto head_of = [&](int t) { return g * G + t / n_qt; };
    auto qtile_of = [&](int t) { return (i_begin + t % n_qt) * kB; };  // first query of step t's tile

    if (warp == 0) {
        // ---------------------------------- producer -------------------------------------
        if (lane == 0) {
            prefetch_tmap(&tq);
            prefetch_tmap(&tk);
            prefetch_tmap(&tv);
            prefetch_tmap(&tdo);
            prefetch_tmap(&tqh);
            prefetch_tmap(&tdoh);
            // resident K_c (B operand of dQ_c = dS K_c)
            mbar_expect_tx(smem_u32(kc_full), 2 * kSub);
            tma_load_4d(sKc, &tk, smem_u32(kc_full), c0, g, krow, bcoord);
            tma_load_4d(sKc + kSub, &tk, smem_u32(kc_full), c0 + 64, g, krow, bcoord);
            int slot = 0, round = 0;
            auto next = [&](uint32_t& dst, uint32_t& fb) -> bool {
                if (round > 0 && !mbar_wait(smem_u32(&empty[slot]), (round - 1) & 1, abort_flag, a.status, 0x21))
                    return false;
                fb = smem_u32(&full[slot]);
                mbar_expect_tx(fb, kSlot);
                dst = sRing + slot * kSlot;
                if (++slot == C::kStages) slot = 0, ++round;
                return true;
            };
            const CUtensorMap* X = s_role ? &tk : &tv;    // role B operand: the key tile, full width
            const CUtensorMap* Y = s_role ? &tqh : &tdoh; // role A operand: this share's query rows
            // per 64-column sub-tile u: X_u (128 keys), then Y_u = the share's 64 rows of both
            // steps stacked (an absent second step repeats the first; its result is unused)
            auto load_role = [&](int T, int u_begin, int u_end) -> bool {
                const int t0 = 2 * T, t1 = min(2 * T + 1, n - 1);
                const int h0 = head_of(t0), h1 = head_of(t1);
                const int y0 = seq_start + qtile_of(t0) + share * C::NQ, y1 = seq_start + qtile_of(t1) + share * C::NQ;
                for (int u = u_begin; u < u_end; ++u) {
                    uint32_t dst, fb;
                    if (!next(dst, fb)) return false;
                    tma_load_4d(dst, X, fb, 64 * u, g, krow, bcoord);
                    if (!next(dst, fb)) return false;
                    tma_load_4d(dst, Y, fb, 64 * u, h0, y0, bcoord);
                    tma_load_4d(dst + C::NQ * 128, Y, fb, 64 * u, h1, y1, bcoord);
                }
                return true;
            };
            auto load_grad = [&](int t) -> bool {  // B operands of dV_c and dK_c
                const int h = head_of(t), qrow = seq_start + qtile_of(t);
                for (int e = 0; e < 2; ++e) {
                    uint32_t dst, fb;
                    if (!next(dst, fb)) return false;
                    tma_load_4d(dst, &tdo, fb, c0 + 64 * e, h, qrow, bcoord);
                }
                for (int e = 0; e < 2; ++e) {
                    uint32_t dst, fb;
                    if (!next(dst, fb)) return false;
                    tma_load_4d(dst, &tq, fb, c0 + 64 * e, h, qrow, bcoord);
                }
                return true;
            };
            // (No L2 prefetch of future Q / dO tiles: issued two to five steps ahead it made the
            // kernel 3.6 % slower at the dense workload and 11 % slower on packed sequences.)
            // consumption order of the UMMA issuer: role(0) | first half of role(T+1), grad(2T),
            // second half of role(T+1), grad(2T+1) | ...
            constexpr int kHalfU = C::NSUB / 2;
            bool ok = load_role(0, 0, C::NSUB);
            for (int T = 0; ok && T < np; ++T) {
                const bool more = T + 1 < np;
                if (more) ok = load_role(T + 1, 0, kHalfU);
                ok = ok && load_grad(2 * T);
                if (ok && more) ok = load_role(T + 1, kHalfU, C::NSUB);
                if (2 * T + 1 < n) ok = ok && load_grad(2 * T + 1);
            }
            const int issued = round * C::kStages + slot;
            for (int s = 0; s < C::kStages && s < issued; ++s) {
                const int last = s + ((issued - 1 - s) / C::kStages) * C::kStages;
                mbar_drain(smem_u32(&full[s]), (last / C::kStages) & 1, a.status, 0x27);
            }
            mbar_drain(smem_u32(kc_full), 0, a.status, 0x2e);
        }
    } else if (warp == 1) {
        // --------------------------------- UMMA issuer -----------------------------------
        if (lane == 0) {
            constexpr uint32_t idRole = idesc_bf16_f32(128, 128, false, false);  // query rows x key tile
            constexpr uint32_t idG128 = idesc_bf16_f32(128, 128, true, true);    // P^T / dS^T x slice, MN-major
            constexpr uint32_t idG64 = idesc_bf16_f32(128, 64, true, true);      // the same, one 64-column half
            constexpr uint32_t idQ = idesc_bf16_f32(128, 128, false, true);      // dS (K-major) x K_c (N-major)
            const uint16_t mask_s = (uint16_t)((1u << C::NHALF) - 1u);       // writers of P
            const uint16_t mask_d = (uint16_t)(mask_s << C::NHALF);          // writers of dS
            int slot = 0, round = 0;
            auto acquire = [&](uint32_t& addr, int& s) -> bool {
                if (!mbar_wait(smem_u32(&full[slot]), round & 1, abort_flag, a.status, 0x22)) return false;
                tc_fence_after();
                addr = sRing + slot * kSlot;
                s = slot;
                if (++slot == C::kStages) slot = 0, ++round;
                return true;
            };
            // S (or dP) rows of pair-step T: A = the stacked query rows (K-major), B = the key tile
            auto role = [&](int T, int u_begin, int u_end) -> bool {
                if (T > 0 && u_begin == 0) {
                    if (!mbar_wait(smem_u32(r_free), (T - 1) & 1, abort_flag, a.status, 0x29)) return false;
                    tc_fence_after();
                }
                for (int u = u_begin; u < u_end; ++u) {
                    uint32_t xa, ya;
                    int xs, ys;
                    if (!acquire(xa, xs) || !acquire(ya, ys)) return false;
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        umma_bf16_ss(tR, sdesc_sw128(ya + kk * 32, 16, 1024), sdesc_sw128(xa + kk * 32, 16, 1024),
                                     idRole, (u | kk) ? 1u : 0u);
                    umma_commit(smem_u32(&empty[xs]));
                    umma_commit(smem_u32(&empty[ys]));
                }
                if (u_end == C::NSUB) umma_commit(smem_u32(r_full));
                return true;
            };
            // acc += A^T x B over a step's 128 queries: A^T read MN-major from a [128 queries x 128 keys]
            // tile (two 64-key sub-tiles), B = one 128-column slice held as two 64-column ring
            // sub-tiles (N-major); one N = 128 product per K step when they sit in adjacent slots
            auto grad_pair = [&](uint32_t dacc, uint32_t sa, bool acc_in) -> bool {
                uint32_t b0, b1;
                int s0, s1;
                if (!acquire(b0, s0) || !acquire(b1, s1)) return false;
                if (s1 == s0 + 1) {
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk)
                        umma_bf16_ss(dacc, sdesc_sw128(sa + kk * 2048, kSub, 1024), sdesc_sw128(b0 + kk * 2048, kSlot, 1024),
                                     idG128, (acc_in || kk > 0) ? 1u : 0u);
                } else {
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk) {
                        const uint64_t ad = sdesc_sw128(sa + kk * 2048, kSub, 1024);
                        const uint32_t accf = (acc_in || kk > 0) ? 1u : 0u;
                        umma_bf16_ss(dacc, ad, sdesc_sw128(b0 + kk * 2048, kSub, 1024), idG64, accf);
                        umma_bf16_ss(dacc + 64, ad, sdesc_sw128(b1 + kk * 2048, kSub, 1024), idG64, accf);
                    }
                }
                umma_commit(smem_u32(&empty[s0]));
                umma_commit(smem_u32(&empty[s1]));
                return true;
            };
            auto grads = [&](int t) -> bool {
                const int pb = t & 1;
                if (!mbar_wait(smem_u32(&p_full[pb]), (t >> 1) & 1, abort_flag, a.status, 0x23)) return false;
                tc_fence_after();
                mbar_expect_tx(smem_u32(&p_full[pb]), p_rem);  // arm the buffer's next use
                if (!grad_pair(tDV, sP + pb * 2 * kSub, t > 0)) return false;  // dV_c += P^T dO_c
                // an S-role CTA is done with P(t) here; a dP-role CTA also reads it in its
                // elementwise warps (to form dS(t)), so it releases the buffer once they have
                // (released after the dS products instead, the kernel measured 0.6 % slower)
                if (!s_role && !mbar_wait(smem_u32(&p_read[pb]), (t >> 1) & 1, abort_flag, a.status, 0x34)) return false;
                umma_commit_multicast(smem_u32(&p_free[pb]), mask_s);
                if (!mbar_wait(smem_u32(ds_full), t & 1, abort_flag, a.status, 0x24)) return false;
                tc_fence_after();
                mbar_expect_tx(smem_u32(ds_full), ds_rem);
                if (!grad_pair(tDK, sDS, t > 0)) return false;  // dK_c += dS^T Q_c
                if (t == 0 && !mbar_wait(smem_u32(kc_full), 0, abort_flag, a.status, 0x2d)) return false;
                if (t > 0 && !mbar_wait(smem_u32(dq_free), (t - 1) & 1, abort_flag, a.status, 0x25)) return false;
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)  // dQ_c = dS K_c: queries on lanes, K = keys
                    umma_bf16_ss(tDQ, sdesc_sw128(sDS + (kk >> 2) * kSub + (kk & 3) * 32, 16, 1024),
                                 sdesc_sw128(sKc + kk * 2048, kSub, 1024), idQ, kk > 0 ? 1u : 0u);
                umma_commit(smem_u32(dq_full));
                umma_commit_multicast(smem_u32(ds_free), mask_d);
                return true;
            };
            constexpr int kHalfU = C::NSUB / 2;
            bool ok = role(0, 0, C::NSUB);
            for (int T = 0; ok && T < np; ++T) {
                const bool more = T + 1 < np;
                if (more) ok = role(T + 1, 0, kHalfU);
                ok = ok && grads(2 * T);
                if (ok && more) ok = role(T + 1, kHalfU, C::NSUB);
                if (2 * T + 1 < n) ok = ok && grads(2 * T + 1);
            }
            umma_commit(smem_u32(mma_idle));
            mbar_drain(smem_u32(mma_idle), 0, a.status, 0x28);
        }
    } else {
        // ------------------------- elementwise / dQ readout warps ----------------------------
        // Thread j = TMEM lane j of the role result: rows 0..63 belong to step 2T, rows 64..127 to
        // step 2T + 1; within a step, row r is query share * 64 + r of the step's tile. For the
        // dQ readout thread j is query row j of the step's tile; for dV / dK, key row j.
        const int quad = warp & 3;
        const int j = quad * 32 + lane;
        const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
        const int half = quad >> 1;              // which step of the pair this thread's row belongs to
        const int trow = share * C::NQ + (j & 63);  // its row within that step's [128 x 128] tile
        const int kabs = k0 + j;                 // key row (epilogue)
        bool ok = true;

        // dQ_c(t) rows (queries on lanes): scale, stage 32 columns at a time in shared memory
        // and add into the fp32 accumulator with TMA bulk reduce-adds.
        auto drain_dq = [&](int t) -> bool {
            bool w = __all_sync(0xffffffffu, mbar_wait(smem_u32(dq_full), t & 1, abort_flag, a.status, 0x26));
            tc_fence_after();
            const int h = head_of(t);
            const int q0 = qtile_of(t);
            const float f = (q0 + j < L) ? a.scale : 0.f;  // rows past the sequence end add zeros
#pragma unroll 1
            for (int c4 = 0; c4 < 4; ++c4) {
                if (tid == 64) bulk_wait_group_read0();  // the reduce that last read the buffer is done
                named_bar_sync(2, 128);
                if (w) {
                    uint32_t rq[32];
                    tmem_ld32(tDQ + c4 * 32 + lane_base, rq);
                    tmem_ld_wait();
#pragma unroll
                    for (int ch = 0; ch < 8; ++ch)
                        st_shared_v4(sStage + j * 128 + (((uint32_t)ch ^ (uint32_t)(j & 7)) << 4),
                                     __float_as_uint(__uint_as_float(rq[4 * ch]) * f),
                                     __float_as_uint(__uint_as_float(rq[4 * ch + 1]) * f),
                                     __float_as_uint(__uint_as_float(rq[4 * ch + 2]) * f),
                                     __float_as_uint(__uint_as_float(rq[4 * ch + 3]) * f));
                }
                fence_proxy_async_smem();
                w = named_bar_and(2, 128, w);
                if (w && tid == 64) {
                    tma_reduce_add_4d(&tdq, sStage, c0 + 32 * c4, h, seq_start + q0, bcoord);
                    bulk_commit_group();
                }
            }
            tc_fence_before();
            mbar_arrive(smem_u32(dq_free));
            return w;
        };

        // this thread's row of the share -> the step's tile, then the warp's 32 rows to every peer
        auto send = [&](const uint32_t (&pk)[64], uint32_t dst, uint32_t fbar) {
#pragma unroll
            for (int hh = 0; hh < 2; ++hh)
#pragma unroll
                for (int ch = 0; ch < 8; ++ch)
                    st_shared_v4(dst + hh * kSub + sw128_offset(trow, ch * 8), pk[hh * 32 + ch * 4], pk[hh * 32 + ch * 4 + 1],
                                 pk[hh * 32 + ch * 4 + 2], pk[hh * 32 + ch * 4 + 3]);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                const uint32_t row0 = (uint32_t)(share * C::NQ + (quad & 1) * 32) * 128;  // the warp's 32 rows
                for (uint32_t peer = 0; peer < (uint32_t)C::NC; ++peer) {
                    if (peer == rank) continue;
#pragma unroll
                    for (int hh = 0; hh < 2; ++hh) {
                        const uint32_t rows = dst + hh * kSub + row0;
                        bulk_copy_to_peer(mapa_shared(rows, peer), rows, 4096, mapa_shared(fbar, peer));
                    }
                }
            }
            mbar_arrive(fbar);
        };

        // Per pair-step: read the role result and hand it back (the next pair-step's product may
        // start), send P (both steps) or dS of the first step, put out dQ of the previous step,
        // send dS of the second step (its buffer is free once the first step's dK / dQ have read
        // it, and that dQ needs the previous step's dQ out of tensor memory), put out dQ of the
        // first step.
        for (int T = 0; T < np; ++T) {
            const int t = 2 * T + half;   // this thread's step
            const bool real = t < n;      // false only for the absent second step of the last pair
            const int q0 = real ? qtile_of(t) : 0;
            const int qa = q0 + trow;     // this thread's query
            float v = 0.f;                // lse in log2 units (+inf past the end: P = 0), or Delta
            if (real) {
                const int h = head_of(t);
                const size_t li = (a.cu_seqlens ? (size_t)h * a.T + seq_start : ((size_t)seq * a.Hq + h) * a.S) + qa;
                v = qa < L ? (s_role ? a.lse[li] * kLog2e : a.delta[li]) : (s_role ? INFINITY : 0.f);
            }
            ok = ok && __all_sync(0xffffffffu, mbar_wait(smem_u32(r_full), T & 1, abort_flag, a.status, 0x2a));
            uint32_t pk[64];  // this row of P or dS over the 128 keys, bf16 pairs
            if (ok) {
                tc_fence_after();
                if (s_role) {
                    // P(query qa, key k0 + c) = exp2(S * scale * log2 e - lse2); on edge tiles only the
                    // keys c_lo .. c_hi are allowed
                    // (c_hi < c_lo when no key of the tile is allowed: every key is masked)
                    const int c_hi = min(kB - 1, min(qa, L - 1) - k0);
                    const int c_lo = a.window > 0 ? max(0, qa - a.window + 1 - k0) : 0;
                    const bool edge = c_lo > 0 || c_hi < kB - 1;
                    uint32_t rr[128];
#pragma unroll
                    for (int c = 0; c < 4; ++c)
                        tmem_ld32(tR + c * 32 + lane_base, *reinterpret_cast<uint32_t(*)[32]>(&rr[c * 32]));
                    tmem_ld_wait();
                    tc_fence_before();
                    mbar_arrive(smem_u32(r_free));
                    auto p_row = [&](auto masked) {
#pragma unroll
                        for (int c = 0; c < 128; c += 2) {
                            float p0 = fast_exp2(fmaf(__uint_as_float(rr[c]), a.scale_log2, -v));
                            float p1 = fast_exp2(fmaf(__uint_as_float(rr[c + 1]), a.scale_log2, -v));
                            if (decltype(masked)::value) {
                                if (c < c_lo || c > c_hi) p0 = 0.f;
                                if (c + 1 < c_lo || c + 1 > c_hi) p1 = 0.f;
                            }
                            pk[c / 2] = pack_bf16x2(p0, p1);
                        }
                    };
                    if (edge) p_row(std::true_type{});
                    else p_row(std::false_type{});
                    // buffer t & 1 was last read at step t - 2
                    if (real && t >= 2)
                        ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&p_free[half]), ((t >> 1) - 1) & 1, abort_flag, a.status, 0x2b));
                    if (real && ok) send(pk, sP + half * 2 * kSub, smem_u32(&p_full[half]));
                } else {
                    // dS = P (dP - Delta), P from the S-role partner's rows. The role result is read
                    // out and handed back first, so the next pair-step's products need not wait for P.
                    uint32_t rr[128];
#pragma unroll
                    for (int c = 0; c < 4; ++c)
                        tmem_ld32(tR + c * 32 + lane_base, *reinterpret_cast<uint32_t(*)[32]>(&rr[c * 32]));
                    tmem_ld_wait();
                    tc_fence_before();
                    mbar_arrive(smem_u32(r_free));
                    if (real) ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&p_full[half]), (t >> 1) & 1, abort_flag, a.status, 0x2c));
                    if (real && ok) {
                        const uint32_t ptile = sP + half * 2 * kSub;
#pragma unroll
                        for (int hh = 0; hh < 2; ++hh)
#pragma unroll
                            for (int ch = 0; ch < 8; ++ch) {
                                uint32_t pw[4];
                                ld_shared_v4(ptile + hh * kSub + sw128_offset(trow, ch * 8), pw[0], pw[1], pw[2], pw[3]);
#pragma unroll
                                for (int e = 0; e < 4; ++e) {
                                    const int c = hh * 64 + ch * 8 + 2 * e;
                                    pk[c / 2] = pack_bf16x2(__uint_as_float(pw[e] << 16) * (__uint_as_float(rr[c]) - v),
                                                            __uint_as_float(pw[e] & 0xffff0000u) * (__uint_as_float(rr[c + 1]) - v));
                                }
                            }
                        mbar_arrive(smem_u32(&p_read[half]));  // this row of P(t) has been read
                    }
                    // the first step's dS: its buffer was last read at step 2T - 1
                    if (half == 0 && real) {
                        if (t > 0) ok = ok && __all_sync(0xffffffffu, mbar_wait(smem_u32(ds_free), (t - 1) & 1, abort_flag, a.status, 0x2f));
                        if (ok) send(pk, sDS, smem_u32(ds_full));
                    }
                }
            }
            if (T > 0) ok = drain_dq(2 * T - 1) && ok;
            if (!s_role && half == 1 && real) {  // the second step's dS, once dK / dQ of the first have read the buffer
                ok = ok && __all_sync(0xffffffffu, mbar_wait(smem_u32(ds_free), (t - 1) & 1, abort_flag, a.status, 0x2f));
                if (ok) send(pk, sDS, smem_u32(ds_full));
            }
            ok = drain_dq(2 * T) && ok;
            ok = named_bar_and(3, 128, ok);
            if (!ok) break;
        }
        if (ok && (n & 1) == 0) ok = drain_dq(n - 1);
        if (tid == 64) bulk_wait_group0();  // every reduce issued by this CTA has landed
        // every arrival owed to this CTA's exchange barriers has landed before it exits
        if (ok) {
            if (s_role) {
                for (int t = max(0, n - 2); t < n; ++t)
                    mbar_drain(smem_u32(&p_free[t & 1]), (t >> 1) & 1, a.status, 0x30);
            }
            else mbar_drain(smem_u32(ds_free), (n - 1) & 1, a.status, 0x31);
        }
        // ---- epilogue: dV_c, dK_c rows (keys on lanes) -> bf16 -----------------------------
        // dq_full of the last step implies every earlier UMMA (all dV/dK updates) is done.
        tc_fence_after();
        ok = __all_sync(0xffffffffu, ok);
        if (ok) {  // warp-uniform: the TMEM loads below are warp collectives
            const bool key_ok = kabs < L;
            const size_t row = (size_t)(a.cu_seqlens ? seq_start + kabs : seq * a.S + kabs) * a.Hkv + g;
            uint16_t* dv_row = a.dV + row * D + c0;
            uint16_t* dk_row = a.dK + row * D + c0;
#pragma unroll 1
            for (int c4 = 0; c4 < 4; ++c4) {
                uint32_t rv[32], rk[32];
                tmem_ld32(tDV + c4 * 32 + lane_base, rv);
                tmem_ld32(tDK + c4 * 32 + lane_base, rk);
                tmem_ld_wait();
                if (key_ok) {
#pragma unroll
                    for (int e = 0; e < 32; e += 8) {
                        uint4 wv, wk;
                        wv.x = pack_bf16x2(__uint_as_float(rv[e]), __uint_as_float(rv[e + 1]));
                        wv.y = pack_bf16x2(__uint_as_float(rv[e + 2]), __uint_as_float(rv[e + 3]));
                        wv.z = pack_bf16x2(__uint_as_float(rv[e + 4]), __uint_as_float(rv[e + 5]));
                        wv.w = pack_bf16x2(__uint_as_float(rv[e + 6]), __uint_as_float(rv[e + 7]));
                        wk.x = pack_bf16x2(__uint_as_float(rk[e]) * a.scale, __uint_as_float(rk[e + 1]) * a.scale);
                        wk.y = pack_bf16x2(__uint_as_float(rk[e + 2]) * a.scale, __uint_as_float(rk[e + 3]) * a.scale);
                        wk.z = pack_bf16x2(__uint_as_float(rk[e + 4]) * a.scale, __uint_as_float(rk[e + 5]) * a.scale);
                        wk.w = pack_bf16x2(__uint_as_float(rk[e + 6]) * a.scale, __uint_as_float(rk[e + 7]) * a.scale);
                        *reinterpret_cast<uint4*>(dv_row + c4 * 32 + e) = wv;
                        *reinterpret_cast<uint4*>(dk_row + c4 * 32 + e) = wk;
                    }
                }
            }
        }
        tc_fence_before();
    }
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tbase, 512);
    }
    // no CTA leaves while a peer may still address its shared memory
    cluster_sync_all();
    if (*abort_flag) {
        // after a give-up a peer's copy into this CTA may still be in flight: let it land
        const uint64_t t0 = globaltimer();
        while (globaltimer() - t0 < 100000ull) __nanosleep(1000);
    }
}

// Delta = rowsum(dO * o) per (row, head) and zero the fp32 dQ accumulator.
// One warp per (row, head); D / 32 elements per lane.
template <int D>
__global__ void __launch_bounds__(256) bwd_prep_kernel(const uint16_t* __restrict__ o, const uint16_t* __restrict__ dO,
                                                       float* __restrict__ delta, float* __restrict__ dq_acc,
                                                       const int32_t* cu_seqlens, int nseq, int S, int T, int Hq,
                                                       long long rows_times_heads) {
    const long long w = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (w >= rows_times_heads) return;
    const long long row = w / Hq;
    const int h = (int)(w % Hq);
    constexpr int E = D / 32;  // 2, 4, 8 or 16 elements per lane
    const uint16_t* orow = o + w * D + lane * E;
    const uint16_t* drow = dO + w * D + lane * E;
    float acc = 0.f;
    auto dot2 = [](uint32_t x, uint32_t y) {
        return __uint_as_float(x << 16) * __uint_as_float(y << 16) +
               __uint_as_float(x & 0xffff0000u) * __uint_as_float(y & 0xffff0000u);
    };
    if constexpr (E >= 8) {
#pragma unroll
        for (int e = 0; e < E; e += 8) {
            const uint4 a = *reinterpret_cast<const uint4*>(orow + e);
            const uint4 b = *reinterpret_cast<const uint4*>(drow + e);
            acc += dot2(a.x, b.x) + dot2(a.y, b.y) + dot2(a.z, b.z) + dot2(a.w, b.w);
        }
    } else if constexpr (E == 4) {
        const uint2 a = *reinterpret_cast<const uint2*>(orow);
        const uint2 b = *reinterpret_cast<const uint2*>(drow);
        acc = dot2(a.x, b.x) + dot2(a.y, b.y);
    } else {
        acc = dot2(*reinterpret_cast<const uint32_t*>(orow), *reinterpret_cast<const uint32_t*>(drow));
    }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    float* dq = dq_acc + w * D + lane * E;
    if constexpr (E >= 4) {
#pragma unroll
        for (int e = 0; e < E; e += 4) *reinterpret_cast<float4*>(dq + e) = make_float4(0.f, 0.f, 0.f, 0.f);
    } else {
        *reinterpret_cast<float2*>(dq) = make_float2(0.f, 0.f);
    }
    if (lane == 0) {
        size_t li;
        if (cu_seqlens) {
            li = (size_t)h * T + row;  // packed rows are token indices
        } else {
            const long long b = row / S, s = row % S;
            li = ((size_t)b * Hq + h) * S + s;
        }
        delta[li] = acc;
    }
    (void)nseq;
}

__global__ void __launch_bounds__(256) bwd_finalize_kernel(const float* __restrict__ acc, uint16_t* __restrict__ dq,
                                                           long long n8) {
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n8; i += (long long)gridDim.x * blockDim.x) {
        const float4 a = reinterpret_cast<const float4*>(acc)[2 * i];
        const float4 b = reinterpret_cast<const float4*>(acc)[2 * i + 1];
        uint4 w;
        w.x = pack_bf16x2(a.x, a.y);
        w.y = pack_bf16x2(a.z, a.w);
        w.z = pack_bf16x2(b.x, b.y);
        w.w = pack_bf16x2(b.z, b.w);
        reinterpret_cast<uint4*>(dq)[i] = w;
    }
}

template <int D>
cudaError_t launch_bwd_t(const BwdLaunch& L, cudaStream_t stream) {
    const long long rh = (long long)L.total_rows * L.Hq;
    {
        const long long threads = rh * 32;
        const unsigned blocks = (unsigned)((threads + 255) / 256);
        const ProfMark m = prof_begin(stream, "bwd_prep");
        bwd_prep_kernel<D><<<blocks, 256, 0, stream>>>(L.o, L.dO, L.delta, L.dq_acc, L.cu_seqlens, L.nseq, L.S,
                                                       L.total_rows, L.Hq, rh);
        prof_end(stream, m);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    if constexpr (D <= 256) {  // one CTA per key tile and 128-column slice, no cluster
        cudaError_t e = launch_bwd_small_main<D>(L, stream);
        if (e != cudaSuccess) return e;
    } else {
        BwdArgs a;
        a.lse = L.lse, a.delta = L.delta, a.dK = L.dK, a.dV = L.dV;
        a.cu_seqlens = L.cu_seqlens, a.status = L.status;
        a.Hq = L.Hq, a.Hkv = L.Hkv, a.S = L.S, a.window = L.window;
        a.T = L.total_rows;
        a.scale = L.scale;
        a.scale_log2 = L.scale * kLog2e;
        constexpr uint32_t kSmem = Cfg<D>::kSmem;
        cudaError_t e = cudaFuncSetAttribute(bwd_main_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmem);
        if (e != cudaSuccess) return e;
        constexpr int NC = Cfg<D>::NC;
        cudaLaunchConfig_t cfg = {};
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = NC;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.gridDim = dim3(L.Hkv * NC, L.nseq, (L.S + kB - 1) / kB);
        cfg.blockDim = dim3(kThreads);
        cfg.dynamicSmemBytes = kSmem;
        cfg.stream = stream;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        const ProfMark m = prof_begin(stream, D == 256 ? "bwd_main_d256" : "bwd_main_d512");
        e = cudaLaunchKernelEx(&cfg, bwd_main_kernel<D>, L.tq, L.tk, L.tv, L.tdo, L.tqh, L.tdoh, L.tdq, a);
        prof_end(stream, m);
        if (e != cudaSuccess) return e;
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    {
        const long long n8 = rh * D / 8;
        const unsigned blocks = (unsigned)std::min<long long>((n8 + 255) / 256, 152LL * 16);
        const ProfMark m = prof_begin(stream, "bwd_finalize");
        bwd_finalize_kernel<<<blocks, 256, 0, stream>>>(L.dq_acc, L.dQ, n8);
        prof_end(stream, m);
        return cudaGetLastError();
    }
}

}  // namespace

cudaError_t launch_bwd(const BwdLaunch& L, cudaStream_t stream) {
    if (L.nseq == 0 || L.S == 0 || L.total_rows == 0) return cudaSuccess;
    if (L.D == 64) return launch_bwd_t<64>(L, stream);
    if (L.D == 128) return launch_bwd_t<128>(L, stream);
    if (L.D == 256) return launch_bwd_t<256>(L, stream);
    if (L.D == 512) return launch_bwd_t<512>(L, stream);
    return cudaErrorInvalidValue;
}

}  // namespace attn
