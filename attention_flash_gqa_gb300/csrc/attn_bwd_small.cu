// Attention backward main kernel for head_dim 64 and 128 (Qwen3-class heads) and, in its "sliced"
// form, for head_dim 256, for the forward in attn_fwd.cu. The same gradient as the cluster kernel
// in attn_bwd.cu (used at D = 512):
//   P  = exp(scale * Q K^T - lse),   dP = dO V^T,   dS = P * (dP - Delta)
//   dV = P^T dO,   dK = scale * dS^T Q,   dQ = scale * dS K
// but with no cluster and no exchange of P^T / dS^T between CTAs: at D <= 128 one CTA's tensor
// memory holds everything a key tile needs; at D = 256 two CTAs per key tile each own a 128-column
// slice of dV / dK / dQ and recompute S^T and dP^T over all of D (1.4x the tensor work of the
// algorithmic count, against the two shared-memory-to-peer exchanges per step of the cluster kernel).
//
// Source: the head_dim 128 attention of "flex_attention + paged KV + CUDA graphs vs vLLM"
// ("Setup": Qwen3-4B heads) trained with the backward the FFPA page describes for its fused
// kernel ("Gemma4 FFPA attention backend support ...": the fused path recomputes P from the
// saved lse instead of materialising S x S).
//
// One CTA = one 128-key tile x one KV head. It keeps K and V resident in shared memory and
// loops over every query head of the GQA group and every query tile that can see its keys
// (causal / window tile skipping), accumulating dV and dK in tensor memory (summed over the
// group without atomics). Per step (head h, query tile i):
//   S^T  = K Q_i^T         (keys on TMEM lanes)       -> region R0
//   dP^T = V dO_i^T                                    -> region R1
//   elementwise warps: P^T = exp2(S^T * scale * log2 e - lse2) written back over R0 as bf16
//   (the A operand of dV straight from tensor memory), then dS^T = P^T (dP^T - Delta) into
//   shared memory (A operand of dK, and, read MN-major, of dQ)
//   dV += P^T dO_i,   dK += dS^T Q_i,   dQ_i = dS K   (queries on lanes; R1 at D = 128)
//   dQ_i leaves tensor memory at once: scaled, staged 32 columns at a time, and added into
//   the fp32 accumulator with TMA bulk reduce-adds.
// Tensor memory (512 columns): D = 128: [0,128) dV, [128,256) dK, [256,384) R0, [384,512) R1
// (dQ reuses R1 once dP^T has been read); D = 64: dV, dK 64 each, R0 and R1 128 each, dQ 64.
// Warp roles (448 threads): warps 0..7 elementwise work (two warps per key row quarter, one per
// half of the 128 score columns, 32 columns at a time; the step's lse and Delta vectors are
// staged in shared memory and read 4 at a time), warps 8..11 read dQ out (thread j owns query
// row j) so the elementwise warps go on to the next step meanwhile, warp 12 TMA producer, warp 13
// UMMA issuer and TMEM owner. The issuer computes dQ before dK, so the readout starts while dK
// runs. Each half of the score columns keeps its P^T (bf16 pairs) in the first 32 columns of its
// own half of R0.
#include <cuda_runtime.h>

#include <type_traits>

#include "attn_internal.h"
#include "ptx.cuh"

namespace attn {
namespace {

constexpr int kB = 128;  // query tile = key tile = 128 rows
// warps 0..7 elementwise (TMEM lane quarter = warp % 4, score-column half = warp / 4), 8..11 dQ
// readout, 12 TMA producer, 13 UMMA issuer
constexpr int kDrainWarp0 = 8, kProducerWarp = 12, kMmaWarp = 13;
constexpr int kThreads = 448;
constexpr int kEw = 256;  // elementwise threads
constexpr uint32_t kSub = 16384;  // 128 rows x 64 bf16, 128-byte swizzle
constexpr float kLog2e = 1.4426950408889634f;

// D: head dim (the contraction of S^T and dP^T); DS: the columns of dV / dK / dQ this CTA owns.
// DS = D (64, 128): K and V resident, one ring slot per Q or dO tile. DS = 128 < D = 256
// ("sliced"): two CTAs per key tile, each recomputing S^T and dP^T over all of D. K stays
// resident (its slice is also dQ's B operand); Q, V and dO stream through the ring as 64-column
// sub-tiles (16 KB slots) in the issuer's order, each released as soon as its product has read
// it. The V / dO pairs stream with the slice's sub-tiles last, so dV reads the slice's dO
// sub-tiles in place (they are the newest slots, so holding them cannot block the strictly
// ordered ring); the slice's Q sub-tiles, needed only after the elementwise step, are streamed
// a second time for dK (held from the S^T stream they would block the ring when it wraps).
// Sliced, one 16 KB dQ staging buffer sits beside a 7-slot ring. (Adding each dQ row straight from
// registers with vector reductions, red.global.add.v4.f32, and giving the buffer to the ring as an
// eighth slot measured 2.77 against 2.68 ms for the window workload's backward; two staging
// buffers and six slots, 2.69 ms.)
template <int D, int DS>
struct SmallCfg {
    static constexpr bool SLICED = DS < D;
    static constexpr int NSUB = D / 64;                   // 64-column sub-tiles of a [128 x D] tile
    static constexpr int NSL = D / DS;                    // CTAs per key tile
    static constexpr uint32_t kTile = NSUB * kSub;        // a whole [128 x D] tile
    static constexpr uint32_t kSlot = SLICED ? kSub : kTile;  // ring slot: a sub-tile (sliced) or a tile
    static constexpr int kStages = SLICED ? 7 : D == 128 ? 3 : 8;
    static constexpr int NSTAGE = SLICED ? 1 : 2;         // dQ staging buffers
    static constexpr bool ALIAS = DS == 128;              // dQ reuses R1
    static constexpr uint32_t kOffK = 0;                  // K tile, resident
    static constexpr uint32_t kOffV = kOffK + kTile;      // V tile, resident (not sliced)
    static constexpr uint32_t kOffDS = kOffV + (SLICED ? 0 : kTile);  // dS^T [128 keys x 128 queries] bf16
    static constexpr uint32_t kOffStage = kOffDS + 2 * kSub;  // dQ staging, NSTAGE x (128 rows x 32 fp32)
    static constexpr uint32_t kOffRing = kOffStage + NSTAGE * kSub;
    static constexpr uint32_t kOffVec = kOffRing + kStages * kSlot;  // step's lse2[128], Delta[128]
    static constexpr uint32_t kOffBar = kOffVec + 1024;
    static constexpr uint32_t kSmem = kOffBar + 512 + 1024;
    static_assert(kSmem <= 232448, "shared memory budget");
};

struct SmallArgs {
    const float* lse;
    const float* delta;
    uint16_t *dK, *dV;
    const int32_t* cu_seqlens;
    unsigned* status;
    int Hq, Hkv, S, window, T;
    float scale, scale_log2;
};

template <int D, int DS>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_small_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                     const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap tdo,
                     const __grid_constant__ CUtensorMap tdq, SmallArgs a) {
    using C = SmallCfg<D, DS>;
    const int g = blockIdx.x / C::NSL;        // KV head
    const int c0 = (blockIdx.x % C::NSL) * DS;  // this CTA's columns of dV, dK, dQ
    const int seq = blockIdx.y;
    const int kv_tile = blockIdx.z;  // tile 0 sees the most queries: launched first
    int seq_start = 0, L = a.S, bcoord = seq;
    if (a.cu_seqlens) {
        seq_start = a.cu_seqlens[seq];
        L = a.cu_seqlens[seq + 1] - seq_start;
        bcoord = 0;
        if (!varlen_seq_ok(seq_start, L, a.T, a.S)) {  // reported; nothing of the slice is touched
            if (threadIdx.x == 0 && blockIdx.x == 0 && kv_tile == 0) atomicOr(a.status, DEVSTAT_BOUNDS);
            return;
        }
    }
    const int k0 = kv_tile * kB;
    if (k0 >= L) return;  // uniform: before any barrier or TMEM use
    const int G = a.Hq / a.Hkv;
    const int q_last = a.window > 0 ? min(L, k0 + kB - 1 + a.window) : L;  // exclusive bound on queries
    const int i_begin = k0 / kB, i_end = (q_last + kB - 1) / kB;
    const int n_qt = i_end - i_begin;
    const int n = G * n_qt;  // steps: (head, query tile)

    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    const uint32_t sK = sbase + C::kOffK, sV = sbase + C::kOffV, sDS = sbase + C::kOffDS;
    const uint32_t sStage = sbase + C::kOffStage, sRing = sbase + C::kOffRing;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
    uint64_t* full = bars;                      // [kStages]
    uint64_t* empty = bars + C::kStages;        // [kStages]
    uint64_t* kv_full = bars + 2 * C::kStages;  // K and V resident
    uint64_t* s_full = kv_full + 1;             // S^T(t) in R0
    uint64_t* dp_full = s_full + 1;             // dP^T(t) in R1
    uint64_t* p_full = dp_full + 1;             // P^T(t) written over R0 (128 threads)
    uint64_t* ds_full = p_full + 1;             // dS^T(t) in shared memory, dP^T(t) read (128 threads)
    uint64_t* ds_free = ds_full + 1;            // dK(t) and dQ(t) have read dS^T(t)
    uint64_t* dq_full = ds_free + 1;            // dQ(t) in tensor memory
    uint64_t* dq_free = dq_full + 1;            // dQ(t) read out (128 threads)
    uint64_t* mma_idle = dq_free + 1;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_idle + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (tid == 0) {
        for (int s = 0; s < C::kStages; ++s) {
            mbar_init(smem_u32(&full[s]), 1);
            mbar_init(smem_u32(&empty[s]), 1);
        }
        mbar_init(smem_u32(kv_full), 1);
        mbar_init(smem_u32(s_full), 1);
        mbar_init(smem_u32(dp_full), 1);
        mbar_init(smem_u32(p_full), kEw);
        mbar_init(smem_u32(ds_full), kEw);
        mbar_init(smem_u32(ds_free), 1);
        mbar_init(smem_u32(dq_full), 1);
        mbar_init(smem_u32(dq_free), 128);
        mbar_init(smem_u32(mma_idle), 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == kMmaWarp) {
        tmem_alloc(smem_u32(tmem_slot), 512);
        tmem_relinquish();
    }
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = *tmem_slot;
    const uint32_t tDV = tbase, tDK = tbase + DS, tR0 = tbase + 2 * DS, tR1 = tR0 + 128;
    const uint32_t tDQ = C::ALIAS ? tR1 : tR1 + 128;
    const int krow = seq_start + k0;
    // TMEM lanes a warp may access: 32 * (warp % 4) ..
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const int j = (warp & 3) * 32 + lane;  // key row (S, dP, dV, dK) or query row (dQ)

    if (warp == kProducerWarp) {
        // ---------------------------------- producer -------------------------------------
        if (lane == 0) {
            prefetch_tmap(&tq);
            prefetch_tmap(&tk);
            prefetch_tmap(&tv);
            prefetch_tmap(&tdo);
            mbar_expect_tx(smem_u32(kv_full), (C::SLICED ? 1 : 2) * C::kTile);
            for (int u = 0; u < C::NSUB; ++u) {
                tma_load_4d(sK + u * kSub, &tk, smem_u32(kv_full), 64 * u, g, krow, bcoord);
                if (!C::SLICED) tma_load_4d(sV + u * kSub, &tv, smem_u32(kv_full), 64 * u, g, krow, bcoord);
            }
            int slot = 0, round = 0;
            bool ok = true;
            // one ring slot: sub-tiles u0 .. u0 + nu - 1 of a [128 x D] tile (rows row0, head hh)
            auto load_slot = [&](const CUtensorMap* map, int hh, int row0, int u0, int nu) -> bool {
                if (round > 0 && !mbar_wait(smem_u32(&empty[slot]), (round - 1) & 1, abort_flag, a.status, 0x41))
                    return false;
                const uint32_t fb = smem_u32(&full[slot]);
                mbar_expect_tx(fb, nu * kSub);
                const uint32_t dst = sRing + slot * C::kSlot;
                for (int u = 0; u < nu; ++u) tma_load_4d(dst + u * kSub, map, fb, 64 * (u0 + u), hh, row0, bcoord);
                if (++slot == C::kStages) slot = 0, ++round;
                return true;
            };
            // sliced: the issuer's order is, for every step t, Q(t), VdO(t) and the slice's Q
            // sub-tiles of step t again; Q(t) = the Q_u (u = 0..), VdO(t) = the V_u dO_u pairs with
            // the slice's pairs last
            auto step_rows = [&](int t, int& hh, int& qrow) {
                hh = g * G + t / n_qt;
                qrow = seq_start + (i_begin + t % n_qt) * kB;
            };
            auto load_q = [&](int t) -> bool {
                int hh, qrow;
                step_rows(t, hh, qrow);
                for (int u = 0; u < C::NSUB; ++u)
                    if (!load_slot(&tq, hh, qrow, u, 1)) return false;
                return true;
            };
            auto load_vdo = [&](int t) -> bool {
                int hh, qrow;
                step_rows(t, hh, qrow);
                for (int i = 0; i < C::NSUB; ++i) {  // the slice's sub-tiles last
                    const int u = (c0 / 64 + DS / 64 + i) % C::NSUB;
                    if (!load_slot(&tv, g, krow, u, 1) || !load_slot(&tdo, hh, qrow, u, 1)) return false;
                }
                return true;
            };
            auto load_qc = [&](int t) -> bool {
                int hh, qrow;
                step_rows(t, hh, qrow);
                for (int u = 0; u < DS / 64; ++u)
                    if (!load_slot(&tq, hh, qrow, c0 / 64 + u, 1)) return false;
                return true;
            };
            for (int t = 0; ok && t < n; ++t) {
                const int h = g * G + t / n_qt, qrow = seq_start + (i_begin + t % n_qt) * kB;
                if (C::SLICED) {
                    ok = load_q(t) && load_vdo(t) && load_qc(t);
                } else {
                    // consumption order of the UMMA issuer: Q(0) dO(0) Q(1) dO(1) ...
                    ok = load_slot(&tq, h, qrow, 0, C::NSUB) && load_slot(&tdo, h, qrow, 0, C::NSUB);
                }
            }
            const int issued = round * C::kStages + slot;
            for (int s = 0; s < C::kStages && s < issued; ++s) {
                const int last = s + ((issued - 1 - s) / C::kStages) * C::kStages;
                mbar_drain(smem_u32(&full[s]), (last / C::kStages) & 1, a.status, 0x47);
            }
            mbar_drain(smem_u32(kv_full), 0, a.status, 0x4e);
        }
    } else if (warp == kMmaWarp && C::SLICED) {
        // ------------------------ UMMA issuer, sliced (D = 256) ---------------------------
        if (lane == 0) {
            constexpr uint32_t idS = idesc_bf16_f32(128, 128, false, false);  // X_u x Y_u^T: both K-major
            constexpr uint32_t idG = idesc_bf16_f32(128, 64, false, true);    // P^T / dS^T x 64 slice columns
            constexpr uint32_t idG128 = idesc_bf16_f32(128, 128, false, true);  // dS^T x the slice, both halves
            constexpr uint32_t idQ128 = idesc_bf16_f32(128, 128, true, true);   // dS x the slice of K, both halves
            int slot = 0, round = 0;
            auto acquire = [&](int& s) -> bool {
                if (!mbar_wait(smem_u32(&full[slot]), round & 1, abort_flag, a.status, 0x42)) return false;
                tc_fence_after();
                s = slot;
                if (++slot == C::kStages) slot = 0, ++round;
                return true;
            };
            const int us0 = c0 / 64;  // the slice's first sub-tile
            // descriptor bases, stepped with sdesc_at in the loops (K-major views: LBO unused;
            // N-major: LBO = the 64-column sub-tile stride)
            const uint64_t dKk = sdesc_sw128(sK, 16, 1024), dKn = sdesc_sw128(sK, kSub, 1024);
            const uint64_t dRk = sdesc_sw128(sRing, 16, 1024), dRn = sdesc_sw128(sRing, kSub, 1024);
            const uint64_t dRn2 = sdesc_sw128(sRing, C::kSlot, 1024);
            const uint64_t dSk = sdesc_sw128(sDS, 16, 1024), dSn = sdesc_sw128(sDS, kSub, 1024);
            auto slot_desc = [&](uint64_t base, int s) { return sdesc_at(base, (uint32_t)s * C::kSlot); };
            // S^T = sum_u K_u (resident) Q_u^T, each Q_u released once read
            auto issue_s = [&]() -> bool {
                for (int u = 0; u < C::NSUB; ++u) {
                    int ys;
                    if (!acquire(ys)) return false;
                    const uint64_t da = sdesc_at(dKk, u * kSub), db = slot_desc(dRk, ys);
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        umma_bf16_ss(tR0, sdesc_at(da, kk * 32), sdesc_at(db, kk * 32), idS, (u | kk) ? 1u : 0u);
                    umma_commit(smem_u32(&empty[ys]));
                }
                umma_commit(smem_u32(s_full));
                return true;
            };
            // dP^T = sum_u V_u dO_u^T, both streamed, the slice's pairs last; the slice's dO
            // sub-tiles are kept (doc) for dV
            int doc[2] = {0, 0};
            auto issue_dp = [&]() -> bool {
                for (int i = 0; i < C::NSUB; ++i) {
                    int xs, ys;
                    if (!acquire(xs) || !acquire(ys)) return false;
                    const uint64_t da = slot_desc(dRk, xs), db = slot_desc(dRk, ys);
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        umma_bf16_ss(tR1, sdesc_at(da, kk * 32), sdesc_at(db, kk * 32), idS, (i | kk) ? 1u : 0u);
                    umma_commit(smem_u32(&empty[xs]));
                    if (i >= C::NSUB - DS / 64) doc[i - (C::NSUB - DS / 64)] = ys;
                    else umma_commit(smem_u32(&empty[ys]));
                }
                umma_commit(smem_u32(dp_full));
                return true;
            };
            bool ok = mbar_wait(smem_u32(kv_full), 0, abort_flag, a.status, 0x43);
            tc_fence_after();
            if (ok) ok = issue_s();   // S^T(0)
            if (ok) ok = issue_dp();  // dP^T(0)
            for (int t = 0; ok && t < n; ++t) {
                // dV_c += P^T dO_c: A = P^T (bf16 pairs over R0), B = the slice's two dO sub-tiles
                ok = mbar_wait(smem_u32(p_full), t & 1, abort_flag, a.status, 0x44);
                if (!ok) break;
                tc_fence_after();
                int b0 = doc[0], b1 = doc[1];
                {
                    const uint64_t db0 = slot_desc(dRn, b0), db1 = slot_desc(dRn, b1);
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk) {
                        const uint32_t at = tR0 + (kk >> 2) * 64 + (kk & 3) * 8;
                        const uint32_t accf = (t > 0 || kk > 0) ? 1u : 0u;
                        umma_bf16_ts(tDV, at, sdesc_at(db0, kk * 2048), idG, accf);
                        umma_bf16_ts(tDV + 64, at, sdesc_at(db1, kk * 2048), idG, accf);
                    }
                }
                umma_commit(smem_u32(&empty[b0]));
                umma_commit(smem_u32(&empty[b1]));
                ok = mbar_wait(smem_u32(ds_full), t & 1, abort_flag, a.status, 0x45);
                if (!ok) break;
                tc_fence_after();
                // dQ_c = dS K_c first (its readout starts while dK runs), into R1; K_c is resident,
                // its two 64-column sub-tiles adjacent: one N = 128 product per K step
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)
                    umma_bf16_ss(tDQ, sdesc_at(dSn, kk * 2048), sdesc_at(dKn, us0 * kSub + kk * 2048), idQ128,
                                 kk > 0 ? 1u : 0u);
                umma_commit(smem_u32(dq_full));
                // dK_c += dS^T Q_c: B = the slice's two Q sub-tiles
                ok = acquire(b0) && acquire(b1);
                if (!ok) break;
                if (b1 == b0 + 1) {  // adjacent ring slots (the ring did not wrap between them): N = 128
                    const uint64_t db = slot_desc(dRn2, b0);
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk)
                        umma_bf16_ss(tDK, sdesc_at(dSk, (kk >> 2) * kSub + (kk & 3) * 32), sdesc_at(db, kk * 2048),
                                     idG128, (t > 0 || kk > 0) ? 1u : 0u);
                } else {
                    const uint64_t db0 = slot_desc(dRn, b0), db1 = slot_desc(dRn, b1);
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk) {
                        const uint64_t ad = sdesc_at(dSk, (kk >> 2) * kSub + (kk & 3) * 32);
                        const uint32_t accf = (t > 0 || kk > 0) ? 1u : 0u;
                        umma_bf16_ss(tDK, ad, sdesc_at(db0, kk * 2048), idG, accf);
                        umma_bf16_ss(tDK + 64, ad, sdesc_at(db1, kk * 2048), idG, accf);
                    }
                }
                umma_commit(smem_u32(&empty[b0]));
                umma_commit(smem_u32(&empty[b1]));
                umma_commit(smem_u32(ds_free));
                if (t + 1 < n) {
                    // S^T(t+1) over R0 (after the dV read of R0: the MMA pipe runs in order). Issued
                    // after dQ(t) / dK(t): issuing it first made the issuer wait for Q(t+1) before
                    // it could start dQ(t), lengthening the dQ -> readout -> dP chain.
                    ok = issue_s();
                    if (!ok) break;
                    // dP^T(t+1) over R1 once dQ(t) has left it
                    ok = mbar_wait(smem_u32(dq_free), t & 1, abort_flag, a.status, 0x48);
                    if (!ok) break;
                    tc_fence_after();
                    ok = issue_dp();
                }
            }
            // every issued UMMA has finished before TMEM may be released
            umma_commit(smem_u32(mma_idle));
            mbar_drain(smem_u32(mma_idle), 0, a.status, 0x49);
        }
    } else if (warp == kMmaWarp) {
        // --------------------------------- UMMA issuer -----------------------------------
        if (lane == 0) {
            constexpr uint32_t idS = idesc_bf16_f32(128, 128, false, false);  // K x Q^T: both K-major
            constexpr uint32_t idG = idesc_bf16_f32(128, D, false, true);     // P^T / dS^T x (dO | Q) N-major
            constexpr uint32_t idQ = idesc_bf16_f32(128, D, true, true);      // dS (MN-major) x K (N-major)
            int slot = 0, round = 0;
            auto acquire = [&](int& s) -> bool {
                if (!mbar_wait(smem_u32(&full[slot]), round & 1, abort_flag, a.status, 0x42)) return false;
                tc_fence_after();
                s = slot;
                if (++slot == C::kStages) slot = 0, ++round;
                return true;
            };
            // acc(128 x 128) = X (resident [keys x D], K-major) x Y^T (ring tile [queries x D], K-major)
            // descriptor bases, stepped with sdesc_at in the loops
            const uint64_t dRk = sdesc_sw128(sRing, 16, 1024), dRn = sdesc_sw128(sRing, kSub, 1024);
            const uint64_t dSk = sdesc_sw128(sDS, 16, 1024), dSn = sdesc_sw128(sDS, kSub, 1024);
            const uint64_t dKn = sdesc_sw128(sK, kSub, 1024);
            auto rows_x_tile = [&](uint32_t dacc, uint32_t x, int ys) {
                const uint64_t dx = sdesc_sw128(x, 16, 1024), dy = sdesc_at(dRk, (uint32_t)ys * C::kSlot);
#pragma unroll
                for (int u = 0; u < C::NSUB; ++u)
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        umma_bf16_ss(dacc, sdesc_at(dx, u * kSub + kk * 32), sdesc_at(dy, u * kSub + kk * 32), idS,
                                     (u | kk) ? 1u : 0u);
            };
            bool ok = mbar_wait(smem_u32(kv_full), 0, abort_flag, a.status, 0x43);
            tc_fence_after();
            int qs = 0, ds = 0;  // ring slots of this step's Q and dO tiles
            if (ok) ok = acquire(qs);
            if (ok) {
                rows_x_tile(tR0, sK, qs);  // S^T(0)
                umma_commit(smem_u32(s_full));
            }
            if (ok) ok = acquire(ds);
            if (ok) {
                rows_x_tile(tR1, sV, ds);  // dP^T(0)
                umma_commit(smem_u32(dp_full));
            }
            for (int t = 0; ok && t < n; ++t) {
                // dV += P^T dO: A = P^T (bf16 pairs over R0), B = dO (N-major)
                ok = mbar_wait(smem_u32(p_full), t & 1, abort_flag, a.status, 0x44);
                if (!ok) break;
                tc_fence_after();
                const uint64_t dob = sdesc_at(dRn, (uint32_t)ds * C::kSlot);
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)  // queries 64h .. 64h+63 of P^T sit at R0 columns 64h .. 64h+31
                    umma_bf16_ts(tDV, tR0 + (kk >> 2) * 64 + (kk & 3) * 8, sdesc_at(dob, kk * 2048), idG,
                                 (t > 0 || kk > 0) ? 1u : 0u);
                umma_commit(smem_u32(&empty[ds]));
                const int qs_t = qs;
                // S^T(t+1) over R0: issued after the P V read of R0 (the MMA pipe runs in order)
                if (t + 1 < n) {
                    ok = acquire(qs);
                    if (!ok) break;
                    rows_x_tile(tR0, sK, qs);
                    umma_commit(smem_u32(s_full));
                }
                ok = mbar_wait(smem_u32(ds_full), t & 1, abort_flag, a.status, 0x45);
                if (!ok) break;
                tc_fence_after();
                // dQ(t) = dS K first, so its readout starts while dK(t) runs: A = dS^T read MN-major
                // (queries contiguous), B = K (N-major)
                if (!C::ALIAS && t > 0) {  // its own columns: the previous dQ has been read out
                    ok = mbar_wait(smem_u32(dq_free), (t - 1) & 1, abort_flag, a.status, 0x46);
                    if (!ok) break;
                    tc_fence_after();
                }
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)
                    umma_bf16_ss(tDQ, sdesc_at(dSn, kk * 2048), sdesc_at(dKn, kk * 2048), idQ, kk > 0 ? 1u : 0u);
                umma_commit(smem_u32(dq_full));
                // dK += dS^T Q: A = dS^T (K-major, shared memory), B = Q (N-major)
                const uint64_t qb = sdesc_at(dRn, (uint32_t)qs_t * C::kSlot);
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)
                    umma_bf16_ss(tDK, sdesc_at(dSk, (kk >> 2) * kSub + (kk & 3) * 32), sdesc_at(qb, kk * 2048), idG,
                                 (t > 0 || kk > 0) ? 1u : 0u);
                umma_commit(smem_u32(&empty[qs_t]));
                umma_commit(smem_u32(ds_free));
                // dP^T(t+1) over R1 (at D = 128 once dQ(t) has left it)
                if (t + 1 < n) {
                    if (C::ALIAS) {
                        ok = mbar_wait(smem_u32(dq_free), t & 1, abort_flag, a.status, 0x48);
                        if (!ok) break;
                        tc_fence_after();
                    }
                    ok = acquire(ds);
                    if (!ok) break;
                    rows_x_tile(tR1, sV, ds);
                    umma_commit(smem_u32(dp_full));
                }
            }
            // every issued UMMA has finished before TMEM may be released
            umma_commit(smem_u32(mma_idle));
            mbar_drain(smem_u32(mma_idle), 0, a.status, 0x49);
        }
    } else if (warp >= kDrainWarp0) {
        // ------------------------------ dQ readout warps -----------------------------------
        // dQ(t) rows (queries on lanes): scale, stage 32 columns at a time in shared memory and add
        // into the fp32 accumulator with TMA bulk reduce-adds
        const bool leader = warp == kDrainWarp0 && lane == 0;
        bool ok = true;
        for (int t = 0; t < n; ++t) {
            ok = ok && __all_sync(0xffffffffu, mbar_wait(smem_u32(dq_full), t & 1, abort_flag, a.status, 0x4a));
            tc_fence_after();
            const int h = g * G + t / n_qt;
            const int q0 = (i_begin + t % n_qt) * kB;
            const float f = (q0 + j < L) ? a.scale : 0.f;  // rows past the sequence end add zeros
            // the whole row into registers first, so dQ's columns are handed back at once (at
            // D = 128 the next dP^T waits for them)
            uint32_t rq[DS];
            if (ok) {
#pragma unroll
                for (int c4 = 0; c4 < DS / 32; ++c4) {
                    uint32_t tmp[32];
                    tmem_ld32(tDQ + c4 * 32 + lane_base, tmp);
#pragma unroll
                    for (int e = 0; e < 32; ++e) rq[c4 * 32 + e] = tmp[e];
                }
                tmem_ld_wait();
            }
            tc_fence_before();
            mbar_arrive(smem_u32(dq_free));
#pragma unroll
            for (int c4 = 0; c4 < DS / 32; ++c4) {
                const uint32_t buf = sStage + (c4 % C::NSTAGE) * kSub;
                if (leader) {  // the reduce that last read `buf` is done
                    if (C::NSTAGE == 2) bulk_wait_group_read1();
                    else bulk_wait_group_read0();
                }
                named_bar_sync(2, 128);
                if (ok) {
#pragma unroll
                    for (int ch = 0; ch < 8; ++ch)
                        st_shared_v4(buf + j * 128 + (((uint32_t)ch ^ (uint32_t)(j & 7)) << 4),
                                     __float_as_uint(__uint_as_float(rq[c4 * 32 + 4 * ch]) * f),
                                     __float_as_uint(__uint_as_float(rq[c4 * 32 + 4 * ch + 1]) * f),
                                     __float_as_uint(__uint_as_float(rq[c4 * 32 + 4 * ch + 2]) * f),
                                     __float_as_uint(__uint_as_float(rq[c4 * 32 + 4 * ch + 3]) * f));
                }
                fence_proxy_async_smem();
                ok = named_bar_and(2, 128, ok);
                if (ok && leader) {
                    tma_reduce_add_4d(&tdq, buf, c0 + 32 * c4, h, seq_start + q0, bcoord);
                    bulk_commit_group();
                }
            }
            if (!ok) break;
        }
        if (leader) bulk_wait_group0();  // every reduce issued by this CTA has landed
    } else {
        // --------------------------- elementwise warps (0..7) --------------------------------
        // warp w: key rows 32 (w % 4) .., score columns (queries) 64 hf .. 64 hf + 63, hf = w / 4
        const int hf = warp >> 2;
        const int kabs = k0 + j;
        const bool key_ok = kabs < L;
        float* vec = reinterpret_cast<float*>(smem + C::kOffVec);  // [0,128) lse2, [128,256) Delta
        bool ok = true;
        // this thread's element of the step's lse / Delta vector, loaded a step ahead
        auto fetch = [&](int t) -> float {
            if (t >= n) return 0.f;
            const int h = g * G + t / n_qt;
            const int qa = (i_begin + t % n_qt) * kB + (tid & 127);
            const size_t lbase = a.cu_seqlens ? (size_t)h * a.T + seq_start : ((size_t)seq * a.Hq + h) * a.S;
            if (tid < 128) return qa < L ? a.lse[lbase + qa] * kLog2e : INFINITY;  // +inf: P = 0 past the end
            return qa < L ? a.delta[lbase + qa] : 0.f;
        };
        float vnext = fetch(0);
        for (int t = 0; t < n; ++t) {
            const int q0 = (i_begin + t % n_qt) * kB;
            vec[tid] = vnext;
            vnext = fetch(t + 1);
            named_bar_sync(3, kEw);
            // ---- P^T = exp2(S^T * scale * log2 e - lse2), written back over R0 as bf16 ----
            // 32 score columns at a time; this half's P columns [64 hf + 16c, +16) overwrite
            // scores of its own first chunk, already read
            ok = ok && __all_sync(0xffffffffu, mbar_wait(smem_u32(s_full), t & 1, abort_flag, a.status, 0x4b));
            uint32_t pk[32];
            if (ok) {
                tc_fence_after();
                const bool edge = !(k0 + kB - 1 <= q0 && (a.window <= 0 || q0 + kB - 1 - k0 < a.window) &&
                                    q0 + kB <= L && k0 + kB <= L);
                // on edge tiles key j sees the queries qa with 0 <= qa - kabs < span
                int qhi = key_ok ? L : kabs;
                if (a.window > 0) qhi = min(qhi, kabs + a.window);
                const unsigned span = qhi > kabs ? (unsigned)(qhi - kabs) : 0u;
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    const int col0 = 64 * hf + 32 * c;  // first query column of the chunk
                    uint32_t rr[32];
                    tmem_ld32(tR0 + col0 + lane_base, rr);
                    tmem_ld_wait();
                    auto p_chunk = [&](auto masked) {
#pragma unroll
                        for (int e = 0; e < 32; e += 4) {
                            const float4 lv = *reinterpret_cast<const float4*>(vec + col0 + e);
                            const float lvs[4] = {lv.x, lv.y, lv.z, lv.w};
                            float p[4];
#pragma unroll
                            for (int u = 0; u < 4; ++u) {
                                p[u] = fast_exp2(fmaf(__uint_as_float(rr[e + u]), a.scale_log2, -lvs[u]));
                                if (decltype(masked)::value && (unsigned)(q0 + col0 + e + u - kabs) >= span) p[u] = 0.f;
                            }
                            pk[16 * c + e / 2] = pack_bf16x2(p[0], p[1]);
                            pk[16 * c + e / 2 + 1] = pack_bf16x2(p[2], p[3]);
                        }
                    };
                    if (edge) p_chunk(std::true_type{});
                    else p_chunk(std::false_type{});
                    uint32_t w[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e) w[e] = pk[16 * c + e];
                    tmem_st16(tR0 + 64 * hf + 16 * c + lane_base, w);
                }
                tmem_st_wait();
                tc_fence_before();
                mbar_arrive(smem_u32(p_full));
            }
            // ---- dS^T = P^T (dP^T - Delta) -> shared memory (sub-tile hf), 32 columns at a time ----
            ok = ok && __all_sync(0xffffffffu, mbar_wait(smem_u32(dp_full), t & 1, abort_flag, a.status, 0x4c));
            if (ok && t > 0) ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(ds_free), (t - 1) & 1, abort_flag, a.status, 0x4d));
            if (ok) {
                tc_fence_after();
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    const int col0 = 64 * hf + 32 * c;
                    uint32_t rr[32];
                    tmem_ld32(tR1 + col0 + lane_base, rr);
                    tmem_ld_wait();
#pragma unroll
                    for (int ch = 0; ch < 4; ++ch) {  // 16-byte chunks: 8 queries each
                        const float4 d0 = *reinterpret_cast<const float4*>(vec + 128 + col0 + 8 * ch);
                        const float4 d1 = *reinterpret_cast<const float4*>(vec + 128 + col0 + 8 * ch + 4);
                        const float dv[8] = {d0.x, d0.y, d0.z, d0.w, d1.x, d1.y, d1.z, d1.w};
                        uint32_t out[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int cc = ch * 8 + 2 * e;  // column within the 32-column chunk
                            const uint32_t pw = pk[16 * c + cc / 2];
                            out[e] = pack_bf16x2(__uint_as_float(pw << 16) * (__uint_as_float(rr[cc]) - dv[2 * e]),
                                                 __uint_as_float(pw & 0xffff0000u) * (__uint_as_float(rr[cc + 1]) - dv[2 * e + 1]));
                        }
                        st_shared_v4(sDS + hf * kSub + sw128_offset(j, 32 * c + 8 * ch), out[0], out[1], out[2], out[3]);
                    }
                }
                fence_proxy_async_smem();
                tc_fence_before();
                mbar_arrive(smem_u32(ds_full));
            }
            ok = named_bar_and(3, kEw, ok);  // also: every read of vec for this step is done
            if (!ok) break;
        }
        // ---- epilogue: dV, dK rows (keys on lanes) -> bf16 ------------------------------------
        // the last step's dq_full (below) follows every dV / dK product of the CTA
        if (ok) ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(dq_full), (n - 1) & 1, abort_flag, a.status, 0x4f));
        tc_fence_after();
        ok = __all_sync(0xffffffffu, ok);
        if (ok) {  // warp-uniform: the TMEM loads below are warp collectives
            // dq_full(n-1) was committed after dQ(n-1) but before dK(n-1): wait for the idle
            // commit of the UMMA issuer instead, which follows every product
            ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(mma_idle), 0, abort_flag, a.status, 0x50));
            tc_fence_after();
        }
        if (ok) {
            const size_t row = (size_t)(a.cu_seqlens ? seq_start + kabs : seq * a.S + kabs) * a.Hkv + g;
            uint16_t* dv_row = a.dV + row * D + c0;
            uint16_t* dk_row = a.dK + row * D + c0;
#pragma unroll 1
            for (int c4 = hf; c4 < DS / 32; c4 += 2) {  // the two warps of a lane quarter split the columns
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
    if (warp == kMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tbase, 512);
    }
}

}  // namespace

template <int D>
cudaError_t launch_bwd_small_main(const BwdLaunch& L, cudaStream_t stream) {
    constexpr int DS = D < 128 ? D : 128;
    SmallArgs a;
    a.lse = L.lse, a.delta = L.delta, a.dK = L.dK, a.dV = L.dV;
    a.cu_seqlens = L.cu_seqlens, a.status = L.status;
    a.Hq = L.Hq, a.Hkv = L.Hkv, a.S = L.S, a.window = L.window, a.T = L.total_rows;
    a.scale = L.scale, a.scale_log2 = L.scale * kLog2e;
    constexpr uint32_t kSmem = SmallCfg<D, DS>::kSmem;
    cudaError_t e =
        cudaFuncSetAttribute(bwd_small_kernel<D, DS>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmem);
    if (e != cudaSuccess) return e;
    const dim3 grid(L.Hkv * (D / DS), L.nseq, (L.S + kB - 1) / kB);
    const ProfMark m = prof_begin(stream, D == 256 ? "bwd_main_d256" : D == 128 ? "bwd_main_d128" : "bwd_main_d64");
    bwd_small_kernel<D, DS><<<grid, kThreads, kSmem, stream>>>(L.tq, L.tk, L.tv, L.tdo, L.tdq, a);
    prof_end(stream, m);
    return cudaGetLastError();
}

template cudaError_t launch_bwd_small_main<64>(const BwdLaunch&, cudaStream_t);
template cudaError_t launch_bwd_small_main<128>(const BwdLaunch&, cudaStream_t);
template cudaError_t launch_bwd_small_main<256>(const BwdLaunch&, cudaStream_t);

}  // namespace attn
