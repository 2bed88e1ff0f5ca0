// Attention backward on tcgen05 tensor cores (D = 256 or 512), for the forward in
// attn_fwd.cu. Given dO, lse and Delta = rowsum(dO * o):
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
//  2. bwd_main: one CTA per (KV tile of 128 keys, KV head, 128-wide slice of D). It
//     loops over every query head of the GQA group and every query tile that can see
//     its keys (causal / window tile skipping), so dK and dV are summed over the group
//     in tensor memory without atomics. Tensor memory (512 columns):
//       [0, 128)   S = Q K^T (queries on lanes); reused for the dQ slice dS K_c
//       [128, 256) dP = dO V^T; the softmax warps move dP(t) into registers first, so
//                  the MMA can compute dP(t+1) while they work on step t
//       [256, 384) dV_c accumulator (keys on lanes), [384, 512) dK_c accumulator
//     S and dP contract over the full D, so each of the D/128 slice CTAs recomputes
//     them; dV_c, dK_c and dQ_c are each computed once. dQ_c leaves TMEM after every
//     query tile and is added into the fp32 accumulator with vector atomics.
//     The softmax warps write P and dS (bf16) to shared memory; the same tiles serve
//     as the MN-major A operand of P^T dO_c / dS^T Q_c and the K-major A of dS K_c.
//  3. bwd_finalize: dQ accumulator -> bf16.
#include <cuda_runtime.h>

#include <algorithm>

#include "attn_internal.h"
#include "ptx.cuh"

namespace attn {
namespace {

constexpr int kB = 128;  // query tile = key tile = 128 rows
constexpr int kThreads = 192;
constexpr uint32_t kSlotBytes = 32768;
constexpr uint32_t kSubBytes = 16384;
constexpr int kStages = 5;
constexpr uint32_t kOffP = kStages * kSlotBytes;
constexpr uint32_t kOffDS = kOffP + kSlotBytes;
constexpr uint32_t kOffBar = kOffDS + kSlotBytes;
constexpr uint32_t kSmem = kOffBar + 256 + 1024;

struct BwdArgs {
    const float* lse;
    const float* delta;
    float* dq_acc;
    uint16_t *dK, *dV;
    const int32_t* cu_seqlens;
    unsigned* status;
    int Hq, Hkv, S, D, window, n_kvtiles, nslices, T;
    float scale, scale_log2;
};

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_main_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                    const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap tdo,
                    const __grid_constant__ CUtensorMap tdq, BwdArgs a) {
    constexpr int kChunks = D / 128;  // 32 KB slots per full-width row tile
    const int g = blockIdx.x / a.nslices, cs = blockIdx.x % a.nslices;
    const int seq = blockIdx.y;
    const int kv_tile = blockIdx.z;  // tile 0 sees the most queries: launched first
    int seq_start = 0, L = a.S, bcoord = seq;
    if (a.cu_seqlens) {
        seq_start = a.cu_seqlens[seq];
        L = a.cu_seqlens[seq + 1] - seq_start;
        bcoord = 0;
    }
    const int k0 = kv_tile * kB;
    if (k0 >= L) return;
    const int G = a.Hq / a.Hkv;
    const int q_last = a.window > 0 ? min(L, k0 + kB - 1 + a.window) : L;  // exclusive bound on queries
    const int i_begin = k0 / kB, i_end = (q_last + kB - 1) / kB;
    const int n_qt = i_end - i_begin;
    const int n = G * n_qt;  // steps: (head, query tile)
    const int c0 = cs * 128;  // this CTA's column slice of D

    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    const uint32_t sSlots = sbase, sP = sbase + kOffP, sDS = sbase + kOffDS;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBar);
    uint64_t* full = bars;
    uint64_t* empty = bars + kStages;
    uint64_t* s_full = bars + 2 * kStages;  // S(t) complete
    uint64_t* dp_full = s_full + 1;          // dP(t) complete
    uint64_t* dp_free = dp_full + 1;         // dP(t) read out of TMEM by the softmax warps
    uint64_t* p_full = dp_free + 1;
    uint64_t* dq_full = p_full + 1;
    uint64_t* dq_free = dq_full + 1;
    uint64_t* stage_full = dq_free + 1;   // all 128 dQ rows staged in smem
    uint64_t* stage_free = stage_full + 1; // the previous step's reduce has read the staging smem
    uint64_t* mma_idle = stage_free + 1;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_idle + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(smem_u32(&full[s]), 1);
            mbar_init(smem_u32(&empty[s]), 1);
        }
        mbar_init(smem_u32(s_full), 1);
        mbar_init(smem_u32(dp_full), 1);
        mbar_init(smem_u32(dp_free), 128);
        mbar_init(smem_u32(p_full), 128);
        mbar_init(smem_u32(dq_full), 1);
        mbar_init(smem_u32(dq_free), 128);
        mbar_init(smem_u32(stage_full), 128);
        mbar_init(smem_u32(stage_free), 1);
        mbar_init(smem_u32(mma_idle), 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), 512);
        tmem_relinquish();
    }
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = *tmem_slot;
    const uint32_t tS = tbase, tDP = tbase + 128, tDV = tbase + 256, tDK = tbase + 384;
    const int krow = seq_start + k0;

    if (warp == 0) {
        // ---------------------------------- producer -------------------------------------
        if (lane == 0) {
            prefetch_tmap(&tq);
            prefetch_tmap(&tk);
            prefetch_tmap(&tv);
            prefetch_tmap(&tdo);
            int slot = 0, round = 0;
            auto load = [&](const CUtensorMap* map, int head, int col0, int row0) -> bool {
                if (round > 0 && !mbar_wait(smem_u32(&empty[slot]), (round - 1) & 1, abort_flag, a.status, 0x21)) return false;
                const uint32_t fb = smem_u32(&full[slot]);
                mbar_expect_tx(fb, kSlotBytes);
                const uint32_t dst = sSlots + slot * kSlotBytes;
                tma_load_4d(dst, map, fb, col0, head, row0, bcoord);
                tma_load_4d(dst + kSubBytes, map, fb, col0 + 64, head, row0, bcoord);
                if (++slot == kStages) slot = 0, ++round;
                return true;
            };
            auto load_dp = [&](int t) -> bool {  // dP = dO V^T operands, chunk pairs
                const int h = g * G + t / n_qt, qrow = seq_start + (i_begin + t % n_qt) * kB;
                for (int c = 0; c < kChunks; ++c) {
                    if (!load(&tdo, h, c * 128, qrow)) return false;
                    if (!load(&tv, g, c * 128, krow)) return false;
                }
                return true;
            };
            auto load_s = [&](int t) -> bool {  // S = Q K^T operands, chunk pairs
                const int h = g * G + t / n_qt, qrow = seq_start + (i_begin + t % n_qt) * kB;
                for (int c = 0; c < kChunks; ++c) {
                    if (!load(&tq, h, c * 128, qrow)) return false;
                    if (!load(&tk, g, c * 128, krow)) return false;
                }
                return true;
            };
            auto load_grad = [&](int t) -> bool {  // B operands of dV_c, dK_c, dQ_c
                const int h = g * G + t / n_qt, qrow = seq_start + (i_begin + t % n_qt) * kB;
                return load(&tdo, h, c0, qrow) && load(&tq, h, c0, qrow) && load(&tk, g, c0, krow);
            };
            // Q and dO tiles are new every step and mostly miss L2 (they are re-read by every
            // key tile of the head group, long after): warm L2 with them two steps ahead so the
            // ring's copies find them there.
            constexpr int kAhead = 2;
            auto prefetch_q_do = [&](int t) {
                if (t >= n) return;
                const int h = g * G + t / n_qt, qrow = seq_start + (i_begin + t % n_qt) * kB;
                for (int c = 0; c < D; c += 64) {
                    tma_prefetch_4d(&tq, c, h, qrow, bcoord);
                    tma_prefetch_4d(&tdo, c, h, qrow, bcoord);
                }
            };
            for (int t = 1; t <= kAhead; ++t) prefetch_q_do(t);
            // the UMMA issuer's consumption order: dP(0) S(0) | dP(t+1) grad(t) S(t+1) | ...
            bool ok = load_dp(0) && load_s(0);
            for (int t = 0; ok && t < n; ++t) {
                prefetch_q_do(t + 1 + kAhead);
                if (t + 1 < n) ok = load_dp(t + 1);
                ok = ok && load_grad(t);
                if (ok && t + 1 < n) ok = load_s(t + 1);
            }
            const int issued = round * kStages + slot;
            for (int s = 0; s < kStages && s < issued; ++s) {
                const int last = s + ((issued - 1 - s) / kStages) * kStages;
                mbar_drain(smem_u32(&full[s]), (last / kStages) & 1, a.status, 0x27);
            }
        }
    } else if (warp == 1) {
        // --------------------------------- UMMA issuer -----------------------------------
        if (lane == 0) {
            constexpr uint32_t idKK = idesc_bf16_f32(128, 128, false, false);  // S, dP, (dQ uses idKN)
            constexpr uint32_t idMN = idesc_bf16_f32(128, 128, true, true);    // dV, dK: A^T and B N-major
            constexpr uint32_t idKN = idesc_bf16_f32(128, 128, false, true);   // dQ: dS K-major, K_c N-major
            int slot = 0, round = 0;
            bool ok = true;
            // Waits for the current slot; on success returns true and its address in `addr`.
            auto acquire = [&](uint32_t& addr) -> bool {
                if (!mbar_wait(smem_u32(&full[slot]), round & 1, abort_flag, a.status, 0x22)) return false;
                tc_fence_after();
                addr = sSlots + slot * kSlotBytes;
                return true;
            };
            auto release = [&]() {
                umma_commit(smem_u32(&empty[slot]));
                if (++slot == kStages) slot = 0, ++round;
            };
            // full-width contraction of two row tiles streamed as (A chunk, B chunk) pairs
            auto contract = [&](uint32_t dst) -> bool {
                for (int c = 0; c < kChunks; ++c) {
                    uint32_t sa, sb;
                    if (!acquire(sa)) return false;
                    const int sa_slot = slot;
                    if (++slot == kStages) slot = 0, ++round;
                    if (!acquire(sb)) return false;
                    for (int sub = 0; sub < 2; ++sub)
                        for (int kk = 0; kk < 4; ++kk) {
                            const uint64_t ad = sdesc_sw128(sa + sub * kSubBytes + kk * 32, 16, 1024);
                            const uint64_t bd = sdesc_sw128(sb + sub * kSubBytes + kk * 32, 16, 1024);
                            umma_bf16_ss(dst, ad, bd, idKK, (c | sub | kk) ? 1u : 0u);
                        }
                    umma_commit(smem_u32(&empty[sa_slot]));
                    release();
                }
                return true;
            };
            ok = contract(tDP);
            if (ok) umma_commit(smem_u32(dp_full));
            ok = ok && contract(tS);
            if (ok) umma_commit(smem_u32(s_full));
            for (int t = 0; ok && t < n; ++t) {
                if (t + 1 < n) {
                    // dP(t+1) overwrites the dP columns as soon as the softmax warps hold dP(t)
                    // in registers, overlapping their work on step t.
                    ok = mbar_wait(smem_u32(dp_free), t & 1, abort_flag, a.status, 0x29);
                    if (!ok) break;
                    tc_fence_after();
                    if (!contract(tDP)) { ok = false; break; }
                    umma_commit(smem_u32(dp_full));
                }
                ok = mbar_wait(smem_u32(p_full), t & 1, abort_flag, a.status, 0x23);
                if (!ok) break;
                tc_fence_after();
                // dV_c += P^T dO_c
                uint32_t sb;
                if (!acquire(sb)) { ok = false; break; }
                for (int kk = 0; kk < 8; ++kk) {
                    const uint64_t ad = sdesc_sw128(sP + kk * 2048, kSubBytes, 1024);
                    const uint64_t bd = sdesc_sw128(sb + kk * 2048, kSubBytes, 1024);
                    umma_bf16_ss(tDV, ad, bd, idMN, (t > 0 || kk > 0) ? 1u : 0u);
                }
                release();
                // dK_c += dS^T Q_c
                if (!acquire(sb)) { ok = false; break; }
                for (int kk = 0; kk < 8; ++kk) {
                    const uint64_t ad = sdesc_sw128(sDS + kk * 2048, kSubBytes, 1024);
                    const uint64_t bd = sdesc_sw128(sb + kk * 2048, kSubBytes, 1024);
                    umma_bf16_ss(tDK, ad, bd, idMN, (t > 0 || kk > 0) ? 1u : 0u);
                }
                release();
                // dQ_c = dS K_c  (into the S columns, already read by the softmax warps)
                if (!acquire(sb)) { ok = false; break; }
                for (int kk = 0; kk < 8; ++kk) {
                    const uint64_t ad = sdesc_sw128(sDS + (kk >> 2) * kSubBytes + (kk & 3) * 32, 16, 1024);
                    const uint64_t bd = sdesc_sw128(sb + kk * 2048, kSubBytes, 1024);
                    umma_bf16_ss(tS, ad, bd, idKN, kk > 0 ? 1u : 0u);
                }
                release();
                umma_commit(smem_u32(dq_full));
                if (t + 1 < n) {
                    // S(t+1) reuses the S columns once dQ(t) has been read out
                    ok = mbar_wait(smem_u32(dq_free), t & 1, abort_flag, a.status, 0x24);
                    if (!ok) break;
                    tc_fence_after();
                    if (!contract(tS)) { ok = false; break; }
                    umma_commit(smem_u32(s_full));
                }
            }
            umma_commit(smem_u32(mma_idle));
            mbar_drain(smem_u32(mma_idle), 0, a.status, 0x28);
        }
    } else {
        // --------------------------- softmax-gradient warps ------------------------------
        const int quad = warp & 3;
        const int r = quad * 32 + lane;
        const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
        bool ok = true;
        uint32_t rdp[128];
        // dP of a step: whole row into registers, then hand the columns back to the MMA
        auto load_dp = [&](int t) -> bool {
            if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(dp_full), t & 1, abort_flag, a.status, 0x2a))) return false;
            tc_fence_after();
#pragma unroll
            for (int c4 = 0; c4 < 4; ++c4) {
                uint32_t tmp[32];
                tmem_ld32(tDP + c4 * 32 + lane_base, tmp);
#pragma unroll
                for (int e = 0; e < 32; ++e) rdp[c4 * 32 + e] = tmp[e];
            }
            tmem_ld_wait();
            tc_fence_before();
            mbar_arrive(smem_u32(dp_free));
            return true;
        };
        if (n > 0) ok = load_dp(0);
        for (int t = 0; ok && t < n; ++t) {
            const int h = g * G + t / n_qt;
            const int q0 = (i_begin + t % n_qt) * kB;
            const int qi = q0 + r;
            const bool row_ok = qi < L;
            float lse2 = INFINITY, dlt = 0.f;
            if (row_ok) {
                const size_t li = a.cu_seqlens ? (size_t)h * a.T + seq_start + qi : ((size_t)seq * a.Hq + h) * a.S + qi;
                lse2 = a.lse[li] * 1.4426950408889634f;
                dlt = a.delta[li];
            }
            // dP(t) is already in registers (loaded right after step t-1's P/dS, or in the
            // prologue below for t = 0), so the MMA can compute dP(t+1) meanwhile.
            ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(s_full), t & 1, abort_flag, a.status, 0x25));
            if (!ok) break;
            tc_fence_after();
            const bool edge = !(k0 + kB - 1 <= q0 && (a.window <= 0 || q0 + kB - 1 - k0 < a.window) && q0 + kB <= L &&
                                k0 + kB <= L);
            if (t > 0) {
                // sP/sdS double as the dQ staging tile of step t-1: wait until its reduce has read it
                if (tid == 64) {
                    bulk_wait_group_read0();
                    mbar_arrive(smem_u32(stage_free));
                }
                ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(stage_free), (t - 1) & 1, abort_flag, a.status, 0x2b));
                if (!ok) break;
            }
#pragma unroll
            for (int c4 = 0; c4 < 4; ++c4) {
                uint32_t rs[32];
                tmem_ld32(tS + c4 * 32 + lane_base, rs);
                tmem_ld_wait();
                uint32_t pk[16], dk[16];
#pragma unroll
                for (int e = 0; e < 32; e += 2) {
                    float p[2], ds[2];
#pragma unroll
                    for (int u = 0; u < 2; ++u) {
                        const int key = k0 + c4 * 32 + e + u;
                        bool allowed = row_ok;
                        if (edge) allowed = allowed && key <= qi && key < L && (a.window <= 0 || qi - key < a.window);
                        const float sv = __uint_as_float(rs[e + u]);
                        p[u] = allowed ? fast_exp2(fmaf(sv, a.scale_log2, -lse2)) : 0.f;
                        ds[u] = p[u] * (__uint_as_float(rdp[c4 * 32 + e + u]) - dlt);
                    }
                    pk[e >> 1] = pack_bf16x2(p[0], p[1]);
                    dk[e >> 1] = pack_bf16x2(ds[0], ds[1]);
                }
                // keys c4*32 .. c4*32+31 -> sub-tile (c4 >> 1), columns (c4 & 1) * 32 ..
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const uint32_t off = (c4 >> 1) * kSubBytes + sw128_offset(r, (c4 & 1) * 32 + u * 8);
                    st_shared_v4(sP + off, pk[4 * u], pk[4 * u + 1], pk[4 * u + 2], pk[4 * u + 3]);
                    st_shared_v4(sDS + off, dk[4 * u], dk[4 * u + 1], dk[4 * u + 2], dk[4 * u + 3]);
                }
            }
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive(smem_u32(p_full));
            // next step's dP first (its columns are then free for dP(t+2)), then the dQ(t) readout
            if (t + 1 < n) {
                ok = load_dp(t + 1);
                if (!ok) break;
            }
            // dQ_c rows: scale and stage in shared memory (the P/dS tiles, free once dQ(t) is
            // done), then one thread adds the tile into the fp32 accumulator with TMA bulk
            // reduce-adds that complete in the background.
            ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(dq_full), t & 1, abort_flag, a.status, 0x26));
            if (!ok) break;
            tc_fence_after();
            const float f = row_ok ? a.scale : 0.f;  // rows past the sequence end add zeros
#pragma unroll 1
            for (int c4 = 0; c4 < 4; ++c4) {
                uint32_t rq[32];
                tmem_ld32(tS + c4 * 32 + lane_base, rq);
                tmem_ld_wait();
                // box c4: columns 32*c4 .. +31 (128 bytes per row), 128-byte swizzle
                const uint32_t box = sP + c4 * kSubBytes;
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const uint32_t addr = box + r * 128 + (((uint32_t)j ^ (uint32_t)(r & 7)) << 4);
                    st_shared_v4(addr, __float_as_uint(__uint_as_float(rq[4 * j]) * f),
                                 __float_as_uint(__uint_as_float(rq[4 * j + 1]) * f),
                                 __float_as_uint(__uint_as_float(rq[4 * j + 2]) * f),
                                 __float_as_uint(__uint_as_float(rq[4 * j + 3]) * f));
                }
            }
            tc_fence_before();
            mbar_arrive(smem_u32(dq_free));
            fence_proxy_async_smem();
            mbar_arrive(smem_u32(stage_full));
            if (tid == 64) {
                ok = mbar_wait(smem_u32(stage_full), t & 1, abort_flag, a.status, 0x2c);
                if (ok) {
                    const int qrow = a.cu_seqlens ? seq_start + q0 : q0;
                    for (int c4 = 0; c4 < 4; ++c4)
                        tma_reduce_add_4d(&tdq, sP + c4 * kSubBytes, c0 + 32 * c4, h, qrow, bcoord);
                    bulk_commit_group();
                }
            }
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
        }
        if (tid == 64) bulk_wait_group0();  // every reduce issued by this CTA has landed
        // ---- epilogue: dV_c, dK_c rows (keys on lanes) -> bf16 -----------------------------
        // dq_full of the last step implies every earlier UMMA (all dV/dK updates) is done.
        tc_fence_after();
        const int kj = k0 + r;
        const bool key_ok = kj < L;
        if (ok) {  // warp-uniform: the TMEM loads below are warp collectives
            const size_t row = (size_t)(a.cu_seqlens ? seq_start + kj : seq * a.S + kj) * a.Hkv + g;
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
    constexpr int E = D / 32;  // 8 or 16 elements per lane
    const uint16_t* orow = o + w * D + lane * E;
    const uint16_t* drow = dO + w * D + lane * E;
    float acc = 0.f;
#pragma unroll
    for (int e = 0; e < E; e += 8) {
        const uint4 a = *reinterpret_cast<const uint4*>(orow + e);
        const uint4 b = *reinterpret_cast<const uint4*>(drow + e);
        const uint32_t av[4] = {a.x, a.y, a.z, a.w}, bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            acc += __uint_as_float(av[j] << 16) * __uint_as_float(bv[j] << 16);
            acc += __uint_as_float(av[j] & 0xffff0000u) * __uint_as_float(bv[j] & 0xffff0000u);
        }
    }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    float4* dq = reinterpret_cast<float4*>(dq_acc + w * D + lane * E);
#pragma unroll
    for (int e = 0; e < E / 4; ++e) dq[e] = make_float4(0.f, 0.f, 0.f, 0.f);
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
    {
        BwdArgs a;
        a.lse = L.lse, a.delta = L.delta, a.dq_acc = L.dq_acc, a.dK = L.dK, a.dV = L.dV;
        a.cu_seqlens = L.cu_seqlens, a.status = L.status;
        a.Hq = L.Hq, a.Hkv = L.Hkv, a.S = L.S, a.D = D, a.window = L.window;
        a.n_kvtiles = (L.S + kB - 1) / kB;
        a.nslices = D / 128;
        a.T = L.total_rows;
        a.scale = L.scale;
        a.scale_log2 = L.scale * 1.4426950408889634f;
        cudaError_t e = cudaFuncSetAttribute(bwd_main_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmem);
        if (e != cudaSuccess) return e;
        dim3 grid(L.Hkv * a.nslices, L.nseq, a.n_kvtiles);
        const ProfMark m = prof_begin(stream, D == 256 ? "bwd_main_d256" : "bwd_main_d512");
        bwd_main_kernel<D><<<grid, kThreads, kSmem, stream>>>(L.tq, L.tk, L.tv, L.tdo, L.tdq, a);
        prof_end(stream, m);
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
    if (L.D == 256) return launch_bwd_t<256>(L, stream);
    if (L.D == 512) return launch_bwd_t<512>(L, stream);
    return cudaErrorInvalidValue;
}

}  // namespace attn
