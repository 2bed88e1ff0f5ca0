// Causal / sliding-window attention forward on tcgen05 tensor cores (D = 64, 128, 256 or 512).
//
// Sources: "Gemma4 FFPA attention backend support ..." (operator table: fused
// attention instead of the MATH path that materialises S x S; "Integration": head_dim
// 512 causal attention, dense and varlen paths), and the sliding-window head_dim 256
// layers of "Root cause analysis: Gemma4 sliding-window BF16 cuDNN SDPA NaN on H100".
//
// One CTA computes a 128-query tile of one head against all keys it may see, for one
// 256-wide half of the output columns (D = 512 runs two CTAs per tile, each recomputing
// the full-width scores; D <= 256 runs one). Tensor memory (512 columns x 128 lanes):
//   O accumulator, fp32, row i = lane i: cols [0, 256) (D >= 256), [0, D) otherwise
//   score buffers of 128 columns at the top: two at D >= 256, three at D <= 128 (the issuer
//   then runs two softmax steps ahead). Once a buffer's scores are in registers, the bf16 P
//   tile of that step is written over the first 32 columns of each 64-column half and read
//   from there as the A operand of P V
// Shared memory: the Q tile (resident) and a ring of 32 KB slots (one slot = 128 rows x
// 128 columns of K or V as two 128-byte-swizzled 64-column sub-tiles, filled by TMA):
// 5 slots at D = 256, 3 at D = 512; 16 KB slots of one sub-tile at D = 64.
//
// Warp roles (320 threads):
//   warp 0      TMA producer (one thread): Q once, then K/V slots in MMA order. Over a
//               paged cache the whole warp works: eight lanes fetch one tile's page ids a
//               tile ahead and each issues its page's box into every slot of the tile, and
//               the warp zeroes the last tile's V rows past the sequence end before its P V
//   warp 1      TMEM owner; one thread issues every UMMA and commit
//   warps 2..9  softmax: warps w and w + 4 share query rows 32 (w & 3) .. (TMEM lane quarter
//               w & 3), one thread per row, each warp on one half of the step's 128 keys.
//               Masking, fp32 online softmax in the log2 domain with lazy rescaling (the
//               running max moves only when a tile's max exceeds it by more than 2^8; the
//               pair exchanges its row maxima through shared memory), P -> TMEM, O rescale
//               in TMEM (only then do they wait for the previous P V), and the epilogue
//               (O / l -> bf16, lse), each warp on half of the O columns.
// KV tiles outside the causal / window range are never loaded (tile-granular skipping);
// only tiles that straddle the diagonal, the window edge or the sequence end are masked.
#include <cuda_runtime.h>

#include "attn_internal.h"
#include "ptx.cuh"

namespace attn {
namespace {

constexpr int kBQ = 128, kBKV = 128;
constexpr int kThreads = 320;
constexpr int kSoftmaxThreads = 256;
constexpr uint32_t kSubBytes = 16384;  // 128 rows x 64 bf16
constexpr float kRescaleLog2 = 8.0f;

template <int DQK, bool PAIR = false>
struct FwdCfg {
    static constexpr int kDV = DQK < 256 ? DQK : 256;      // O columns per CTA
    // score buffers in tensor memory: three when O takes at most 128 of the 512 columns, so the
    // issuer runs two softmax steps ahead instead of one
    static constexpr int kSBuf = kDV <= 128 ? 3 : 2;
    static constexpr int kSubs = DQK >= 128 ? 2 : 1;        // 64-column sub-tiles per slot
    static constexpr int kSlotCols = 64 * kSubs;
    static constexpr uint32_t kSlotBytes = kSubs * kSubBytes;
    // A CTA of a pair holds half of each key tile: its 64 keys x 256 columns per slot (four
    // 8 KB sub-tiles of 64 rows), and half of the V columns of the O block: one slot.
    static constexpr int kQChunks = PAIR ? DQK / 256 : DQK / kSlotCols;  // slots per K tile
    static constexpr int kVChunks = PAIR ? 1 : kDV / kSlotCols;          // slots per V tile (this CTA's columns)
    // ring depth: what shared memory leaves next to the resident Q tile
    static constexpr int kStages = DQK == 512 ? 3 : DQK == 256 ? 5 : DQK == 128 ? 6 : 12;
    static constexpr uint32_t kQBytes = DQK * 256;  // 128 rows x DQK bf16
    static constexpr uint32_t kOffSlots = kQBytes;
    static constexpr uint32_t kOffXch = kOffSlots + kStages * kSlotBytes;  // [2 halves][128 rows] fp32
    static constexpr uint32_t kOffBar = kOffXch + 1024;
    static constexpr uint32_t kSmem = kOffBar + 512 + 1024;  // barriers + alignment slack
    // paged slots: the slot's sub-tiles interleaved per 8-row group
    static constexpr uint32_t kPagedGroupStride = 1024 * kSubs;
    // paged K slots of a pair: 64 keys x 256 columns, four 64-column sub-tiles per 8-row group
    static constexpr uint32_t kPairPagedKGroupStride = 4096;
    static_assert(kSmem <= 232448, "shared memory");
    static_assert(!PAIR || DQK >= 256, "the CTA pair serves head_dim 256 and 512");
};

struct FwdArgs {
    uint16_t* o;
    float* lse;
    const int32_t* cu_seqlens;
    unsigned* status;
    int Hq, Hkv, S, D, window, n_qtiles, nsplit, T;
    float scale_log2;
    // paged prefill: keys / values through a block table, new queries packed by cu_q
    const int32_t *block_table, *seq_lens, *cu_q;
    int max_pages, num_pages;
};

// PAGED: chunked prefill over a paged cache ("flex_attention + paged KV + CUDA graphs vs
// vLLM", "Architecture notes": keys and values are read through the block table). A
// sequence is one request: its n new query rows are the last n of its L cached tokens, so
// query index i sits at position L - n + i. Key tile t is 8 pages of 16 tokens. A slot is
// filled by eight 4 KB boxes, one per page: the page's 16 rows x 128 columns of one head,
// taken by a 5-D tensor map over the cache [num_pages, 16, Hkv, D] viewed as
// (64 columns, 8 rows, Hkv*D/64 column chunks, 2 row groups, pages). In shared memory the
// slot then holds 8-row groups of both 64-column chunks interleaved: chunk c of row group G
// (keys 8G .. 8G+7) at byte G*2048 + c*1024, each a 1 KB 128-byte-swizzle atom. The MMA
// descriptors differ only in their strides (kPagedGroupStride); one box moves 256 bytes per
// row, which the TMA engine streams about 1.5x faster than sixteen 16-row boxes of 64 columns.
// PAIR: a cluster of two CTAs (a CTA pair) computes one query tile for two query heads of the
// same GQA group, so both need the same keys and values. The even CTA issues every MMA for
// both as an M = 256 product (tcgen05 cta_group::2): for S = Q K^T each CTA supplies its own Q
// rows and half of the key tile (64 keys), for P V its own P (tensor memory) and half of the
// O block's V columns. Each CTA therefore streams half of K and half of V per key step. Both
// CTAs' copies complete on the even CTA's barriers; the MMA commits are multicast to both; the
// odd CTA's softmax warps report P ready on the even CTA's barrier. Paged and paired, a CTA's
// K slot is its four pages of the key tile, each one 8 KB box of 16 rows x 256 columns (8-row
// groups of four 1 KB sub-tile atoms, 4 KB apart); its V slot is the paged V slot of its 128
// columns. The last tile's V slot, when keys past the end must be zeroed, completes on a
// barrier of its own CTA instead: each CTA zeroes its rows and reports on the even CTA's vfix.
template <int DQK, bool PAGED, bool PAIR>
__global__ void __launch_bounds__(kThreads, 1)
    fwd_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
               const __grid_constant__ CUtensorMap tv, FwdArgs a) {
    using C = FwdCfg<DQK, PAIR>;
    // ---- which tile ------------------------------------------------------------------
    const int h = blockIdx.x;
    const int seq = blockIdx.y / a.nsplit, split = blockIdx.y % a.nsplit;
    const int q_tile = a.n_qtiles - 1 - (int)blockIdx.z;  // longest tiles first
    int seq_start = 0, L = a.S, bcoord = seq;
    int nq = a.S, qoff = 0;  // query rows of the sequence; position of its query row 0
    if (PAGED) {
        seq_start = a.cu_q[seq];
        nq = a.cu_q[seq + 1] - seq_start;
        L = a.seq_lens[seq];
        bcoord = 0;
        if (seq_start < 0 || nq < 0 || nq > a.S || seq_start > a.T - nq || nq > L || L > a.max_pages * 16) {
            // inconsistent request: reported, nothing read or written
            if (threadIdx.x == 0 && split == 0 && h == 0 && q_tile == a.n_qtiles - 1) atomicOr(a.status, DEVSTAT_BOUNDS);
            return;
        }
        qoff = L - nq;
    } else if (a.cu_seqlens) {
        seq_start = a.cu_seqlens[seq];
        L = a.cu_seqlens[seq + 1] - seq_start;
        nq = L;
        bcoord = 0;
        if (!varlen_seq_ok(seq_start, L, a.T, a.S)) {
            // a slice outside the packed rows, or longer than the grid covers: reported, and no
            // row of it is read or written
            if (threadIdx.x == 0 && split == 0 && h == 0 && q_tile == a.n_qtiles - 1) atomicOr(a.status, DEVSTAT_BOUNDS);
            return;
        }
    }
    const int q0 = q_tile * kBQ;
    if (q0 >= nq) return;  // uniform: before any barrier or TMEM use
    const int qp0 = qoff + q0;  // position of the tile's first query
    const int g = h / (a.Hq / a.Hkv);
    const int dv0 = split * C::kDV;
    const int kv_hi = min(L, qp0 + kBQ);
    const int kv_lo = a.window > 0 ? max(0, qp0 - a.window + 1) : 0;
    const int t_begin = kv_lo / kBKV, t_end = (kv_hi + kBKV - 1) / kBKV;
    const int n = t_end - t_begin;

    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    const uint32_t sQ = sbase, sSlots = sbase + C::kOffSlots;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
    uint64_t* full = bars;                     // [kStages]
    uint64_t* empty = bars + C::kStages;       // [kStages]
    uint64_t* q_full = bars + 2 * C::kStages;  // 1
    // per score buffer b (step j uses b = j % kSBuf): one pending phase at most on each, since a
    // buffer's next step cannot start before the issuer has consumed its current one
    uint64_t* s_full = q_full + 1;             // [3]: S(j) in TMEM
    uint64_t* p_full = s_full + 3;             // [3]: P(j) in TMEM (all softmax threads)
    uint64_t* pv_done = p_full + 3;            // [3]: P V(j) complete
    uint64_t* mma_idle = pv_done + 3;          // 1
    uint64_t* vfix = mma_idle + 1;             // 1 (paged): the last tile's V rows past the end are zeroed
    uint64_t* vtail = vfix + 1;                // 1 (paged pair): this CTA's copy of that V slot landed
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(vtail + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    if (tid == 0) {
        for (int s = 0; s < C::kStages; ++s) {
            mbar_init(smem_u32(&full[s]), 1);
            mbar_init(smem_u32(&empty[s]), 1);
        }
        mbar_init(smem_u32(q_full), 1);
        for (int b = 0; b < 3; ++b) mbar_init(smem_u32(&s_full[b]), 1);
        // P ready: every softmax thread, or (pair) one arrival per softmax warp of both CTAs, counted
        // on the even CTA's barrier
        for (int b = 0; b < 3; ++b) mbar_init(smem_u32(&p_full[b]), PAIR ? 2 * kSoftmaxThreads / 32 : kSoftmaxThreads);
        for (int b = 0; b < 3; ++b) mbar_init(smem_u32(&pv_done[b]), 1);
        mbar_init(smem_u32(mma_idle), 1);
        mbar_init(smem_u32(vfix), PAIR ? 2 : 1);
        mbar_init(smem_u32(vtail), 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        if (PAIR) {
            tmem_alloc_pair(smem_u32(tmem_slot), 512);  // the same columns in both CTAs of the pair
            tmem_relinquish_pair();
        } else {
            tmem_alloc(smem_u32(tmem_slot), 512);
            tmem_relinquish();
        }
    }
    __syncthreads();
    if (PAIR) {  // the peer's barriers are initialised before anything signals them
        tc_fence_before();
        cluster_sync_all();
    }
    tc_fence_after();
    const uint32_t tbase = *tmem_slot;
    const uint32_t tO = tbase, tS0 = tbase + 512 - C::kSBuf * 128;
    const uint32_t crank = PAIR ? cluster_ctarank() : 0;  // 0: the CTA that issues the pair's MMAs
    // the even CTA's barriers, in the cluster window (pair: both CTAs' copies complete on them)
    auto lead_bar = [&](const uint64_t* bar) -> uint32_t { return PAIR ? mapa_shared(smem_u32(bar), 0) : smem_u32(bar); };

    // keys past the end in the last tile (paged: their cache rows may hold any bits)
    const bool tail_fix = PAGED && (t_end * kBKV > L);
    if (warp == 0 && PAGED) {
        // -------------------- TMA producer, paged keys / values (whole warp) ---------------
        const int npg = (L + 15) / 16;  // pages of the request
        const int32_t* bt = a.block_table + (size_t)seq * a.max_pages;
        auto page_id = [&](int tile) -> int {  // lane i < 8: id of page i of key tile `tile`
            if (lane >= 8) return 0;
            const int pi = tile * 8 + lane;
            int id = bt[pi < npg ? pi : 0];  // pages past the request: its first page (masked anyway)
            if (id < 0 || id >= a.num_pages) {
                atomicOr(a.status, DEVSTAT_BOUNDS);
                id = 0;
            }
            return id;
        };
        if (lane == 0) {
            prefetch_tmap(&tq);
            prefetch_tmap(&tk);
            prefetch_tmap(&tv);
            if (crank == 0) mbar_expect_tx(smem_u32(q_full), (PAIR ? 2 : 1) * C::kQBytes);
            for (int c = 0; c < DQK / 64; ++c) {
                if (PAIR) tma_load_4d_pair(sQ + c * kSubBytes, &tq, lead_bar(q_full), c * 64, h, seq_start + q0, 0);
                else tma_load_4d(sQ + c * kSubBytes, &tq, smem_u32(q_full), c * 64, h, seq_start + q0, 0);
            }
        }
        int slot = 0, round = 0;
        bool ok = true;
        // one slot = 128 keys x kSlotCols columns: lane i < 8 loads page i's box (16 rows x kSlotCols)
        const int chunk0 = g * (DQK / 64);  // first 64-column chunk of KV head g
        // kind 0: a V slot (lane i < 8: page i, 16 rows x kSlotCols columns); 1: a pair's K slot
        // (lane i < 4: page 4 crank + i, 16 rows x 256 columns); 2: the last V slot of a pair that
        // zeroes keys past the end, completing on this CTA's vtail
        bool vtail_armed = false;
        auto load_slot = [&](const CUtensorMap* map, int col0, int ids, int kind, int& used_slot, int& used_round) -> bool {
            if (round > 0 && !__all_sync(0xffffffffu, mbar_wait(smem_u32(&empty[slot]), (round - 1) & 1, abort_flag,
                                                                 a.status, 0x11)))
                return false;
            const uint32_t dst = sSlots + slot * C::kSlotBytes;
            if (!PAIR) {
                const uint32_t fb = smem_u32(&full[slot]);
                if (lane == 0) mbar_expect_tx(fb, C::kSlotBytes);
                if (lane < 8) tma_load_5d(dst + lane * 2 * C::kPagedGroupStride, map, fb, 0, 0, chunk0 + col0 / 64, 0, ids);
            } else if (kind == 2) {
                // the even CTA's barrier is armed without bytes: the issuer waits for vfix as well
                if (lane == 0) {
                    if (crank == 0) mbar_arrive(smem_u32(&full[slot]));
                    mbar_expect_tx(smem_u32(vtail), C::kSlotBytes);
                }
                vtail_armed = true;
                __syncwarp();
                if (lane < 8)
                    tma_load_5d(dst + lane * 2 * C::kPagedGroupStride, map, smem_u32(vtail), 0, 0, chunk0 + col0 / 64, 0, ids);
            } else {
                const uint32_t fb = lead_bar(&full[slot]);
                if (lane == 0 && crank == 0) mbar_expect_tx(smem_u32(&full[slot]), 2 * C::kSlotBytes);
                if (kind == 1) {
                    const int id = __shfl_sync(0xffffffffu, ids, 4 * (int)crank + (lane & 3));
                    if (lane < 4) tma_load_5d_pair(dst + lane * 2 * C::kPairPagedKGroupStride, map, fb, 0, 0, chunk0 + col0 / 64, 0, id);
                } else if (lane < 8) {
                    tma_load_5d_pair(dst + lane * 2 * C::kPagedGroupStride, map, fb, 0, 0, chunk0 + col0 / 64, 0, ids);
                }
            }
            used_slot = slot, used_round = round;
            if (++slot == C::kStages) slot = 0, ++round;
            return true;
        };
        // page ids one tile ahead, separately for the K and the V sequence
        int k_cur = page_id(t_begin), k_nxt = n > 1 ? page_id(t_begin + 1) : 0;
        int v_cur = k_cur, v_nxt = k_nxt;
        int vs[C::kVChunks], vr[C::kVChunks];
        int kt = 0, vt = 0;  // next K / V tile to load
        auto load_k = [&]() -> bool {
            int us, ur;
            for (int c = 0; c < C::kQChunks; ++c)
                if (!load_slot(&tk, c * (PAIR ? 256 : C::kSlotCols), k_cur, PAIR ? 1 : 0, us, ur)) return false;
            return true;
        };
        auto load_v = [&]() -> bool {
            const int kind = PAIR && tail_fix && vt == n - 1 ? 2 : 0;
            for (int c = 0; c < C::kVChunks; ++c)
                if (!load_slot(&tv, dv0 + (PAIR ? 128 * (int)crank : 0) + c * C::kSlotCols, v_cur, kind, vs[c], vr[c]))
                    return false;
            return true;
        };
        auto next_k = [&]() {
            ++kt;
            k_cur = k_nxt;
            k_nxt = kt + 1 < n ? page_id(t_begin + kt + 1) : 0;
        };
        auto next_v = [&]() {
            ++vt;
            v_cur = v_nxt;
            v_nxt = vt + 1 < n ? page_id(t_begin + vt + 1) : 0;
        };
        // the issuer's order: K(0) .. K(kSBuf - 1), then V(j), K(j + kSBuf) for every step j
        for (int b = 0; ok && b < C::kSBuf && b < n; ++b) {
            ok = load_k();
            next_k();
        }
        for (int j = 0; ok && j < n; ++j) {
            ok = load_v();
            next_v();
            if (ok && j + C::kSBuf < n) {
                ok = load_k();
                next_k();
            }
        }
        if (ok && tail_fix) {
            // zero the rows of keys >= L in the last tile's V slots before their P V (P is 0 there,
            // but 0 * NaN is not 0)
            const int r_valid = L - (t_end - 1) * kBKV;  // 1 .. 127
            if (PAIR) ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(vtail), 0, abort_flag, a.status, 0x1e));
            for (int c = 0; !PAIR && ok && c < C::kVChunks; ++c)
                ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&full[vs[c]]), vr[c] & 1, abort_flag, a.status, 0x1e));
            if (ok) {
                const int units = (kBQ - r_valid) * 8 * C::kSubs;  // 16-byte pieces of the rows past the end
                for (int c = 0; c < C::kVChunks; ++c) {
                    const uint32_t base = sSlots + vs[c] * C::kSlotBytes;
                    for (int e = lane; e < units; e += 32) {
                        const int row = r_valid + e / (8 * C::kSubs), chunk = (e >> 3) % C::kSubs, piece = e & 7;
                        st_shared_v4(base + (row >> 3) * C::kPagedGroupStride + chunk * 1024 + (row & 7) * 128 + piece * 16,
                                     0u, 0u, 0u, 0u);
                    }
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    if (crank == 0) mbar_arrive(smem_u32(vfix));
                    else mbar_arrive_cluster(lead_bar(vfix));
                }
            }
        }
        // pair: the even CTA's barriers count both CTAs' copies (the odd CTA stays until then: the
        // cluster barrier at the end); a vtail copy was waited for above, or is drained here
        if (lane == 0 && crank == 0) {
            const int issued = round * C::kStages + slot;
            for (int s = 0; s < C::kStages && s < issued; ++s) {
                const int last = s + ((issued - 1 - s) / C::kStages) * C::kStages;
                mbar_drain(smem_u32(&full[s]), (last / C::kStages) & 1, a.status, 0x18);
            }
            mbar_drain(smem_u32(q_full), 0, a.status, 0x19);
        }
        if (PAIR && lane == 0 && vtail_armed) mbar_drain(smem_u32(vtail), 0, a.status, 0x1d);
    } else if (warp == 0) {
        // ------------------------------- TMA producer ----------------------------------
        if (lane == 0) {
            prefetch_tmap(&tq);
            prefetch_tmap(&tk);
            prefetch_tmap(&tv);
            const int row_q = seq_start + q0;
            // pair: the even CTA expects both CTAs' bytes on its barriers, and the copies of both
            // complete there
            if (crank == 0) mbar_expect_tx(smem_u32(q_full), (PAIR ? 2 : 1) * C::kQBytes);
            for (int c = 0; c < DQK / 64; ++c) {
                if (PAIR) tma_load_4d_pair(sQ + c * kSubBytes, &tq, lead_bar(q_full), c * 64, h, row_q, bcoord);
                else tma_load_4d(sQ + c * kSubBytes, &tq, smem_u32(q_full), c * 64, h, row_q, bcoord);
            }
            int slot = 0, round = 0;
            bool ok = true;
            // one slot: kSubs sub-tiles of 128 rows x 64 columns (col0 + 64 sub, rows row0 ..); pair
            // K slots: four sub-tiles of 64 rows (this CTA's keys) x 64 columns
            auto load_chunk = [&](const CUtensorMap* map, int col0, int row0, bool k_half) -> bool {
                if (round > 0 && !mbar_wait(smem_u32(&empty[slot]), (round - 1) & 1, abort_flag, a.status, 0x11)) return false;
                if (crank == 0) mbar_expect_tx(smem_u32(&full[slot]), (PAIR ? 2 : 1) * C::kSlotBytes);
                const uint32_t dst = sSlots + slot * C::kSlotBytes;
                if (PAIR) {
                    const uint32_t fb = lead_bar(&full[slot]);
                    if (k_half) {
                        for (int sub = 0; sub < 4; ++sub)
                            tma_load_4d_pair(dst + sub * (kSubBytes / 2), map, fb, col0 + sub * 64, g, row0 + 64 * (int)crank, bcoord);
                    } else {
                        for (int sub = 0; sub < C::kSubs; ++sub)
                            tma_load_4d_pair(dst + sub * kSubBytes, map, fb, col0 + 128 * (int)crank + sub * 64, g, row0, bcoord);
                    }
                } else {
                    const uint32_t fb = smem_u32(&full[slot]);
                    for (int sub = 0; sub < C::kSubs; ++sub)
                        tma_load_4d(dst + sub * kSubBytes, map, fb, col0 + sub * 64, g, row0, bcoord);
                }
                if (++slot == C::kStages) slot = 0, ++round;
                return true;
            };
            auto load_k = [&](int t) -> bool {
                for (int c = 0; c < C::kQChunks; ++c)
                    if (!load_chunk(&tk, c * (PAIR ? 256 : C::kSlotCols), seq_start + (t_begin + t) * kBKV, true)) return false;
                return true;
            };
            auto load_v = [&](int t) -> bool {
                for (int c = 0; c < C::kVChunks; ++c)
                    if (!load_chunk(&tv, dv0 + c * C::kSlotCols, seq_start + (t_begin + t) * kBKV, false)) return false;
                return true;
            };
            // the issuer's order: K(0) .. K(kSBuf - 1), then V(j), K(j + kSBuf) for every step j
            for (int b = 0; ok && b < C::kSBuf && b < n; ++b) ok = load_k(b);
            for (int j = 0; ok && j < n; ++j) {
                ok = load_v(j);
                if (ok && j + C::kSBuf < n) ok = load_k(j + C::kSBuf);
            }
            // Drain: wait (bounded) for the last copy issued into every slot. Pair: the even CTA's
            // barriers count both CTAs' copies, and the odd CTA stays until then (the cluster
            // barrier at the end).
            if (crank == 0) {
                const int issued = round * C::kStages + slot;
                for (int s = 0; s < C::kStages && s < issued; ++s) {
                    const int last = s + ((issued - 1 - s) / C::kStages) * C::kStages;
                    mbar_drain(smem_u32(&full[s]), (last / C::kStages) & 1, a.status, 0x18);
                }
                mbar_drain(smem_u32(q_full), 0, a.status, 0x19);
            }
        }
    } else if (warp == 1) {
        // ------------------------------- UMMA issuer -----------------------------------
        // (pair: the even CTA issues for both; the odd CTA's warp 1 only allocates tensor memory)
        if (lane == 0 && crank == 0) {
            // Q K^T: both K-major (pair: M = 256 over both CTAs' query rows, N = 128 keys split 64 / 64)
            constexpr uint32_t idS = idesc_bf16_f32(PAIR ? 256 : 128, 128, false, false);
            // P (TMEM) V: V is N-major (pair: N = the 256-column O block, 128 columns in each CTA)
            constexpr uint32_t idO = idesc_bf16_f32(PAIR ? 256 : 128, PAIR ? 256 : C::kSlotCols, false, true);
            // a commit reaches this CTA's barrier, or (pair) the barrier at that offset in both CTAs
            auto commit = [&](uint64_t* bar) {
                if (PAIR) umma_commit_pair(smem_u32(bar), (uint16_t)3);
                else umma_commit(smem_u32(bar));
            };
            int slot = 0, round = 0;
            bool ok = mbar_wait(smem_u32(q_full), 0, abort_flag, a.status, 0x12);
            tc_fence_after();
            auto next_slot = [&]() -> bool {
                if (!mbar_wait(smem_u32(&full[slot]), round & 1, abort_flag, a.status, 0x13)) return false;
                tc_fence_after();
                return true;
            };
            auto release_slot = [&]() {
                commit(&empty[slot]);
                if (++slot == C::kStages) slot = 0, ++round;
            };
            // descriptor bases, stepped with sdesc_at in the loops
            const uint64_t dQk = sdesc_sw128(sQ, 16, 1024);
            auto issue_s = [&](int buf) -> bool {
                const uint32_t dst = tS0 + buf * 128;
                for (int c = 0; c < C::kQChunks; ++c) {
                    if (!next_slot()) return false;
                    const uint32_t kslot = sSlots + slot * C::kSlotBytes;
                    if (PAIR) {  // four sub-tiles of this CTA's 64 keys x 64 columns (8 KB each; paged: interleaved)
                        const uint64_t dq = sdesc_at(dQk, 4 * c * kSubBytes);
                        const uint64_t dk = PAGED ? sdesc_sw128(kslot, 16, C::kPairPagedKGroupStride) : sdesc_sw128(kslot, 16, 1024);
#pragma unroll
                        for (int sub = 0; sub < 4; ++sub)
#pragma unroll
                            for (int kk = 0; kk < 4; ++kk)
                                umma_pair_ss(dst, sdesc_at(dq, sub * kSubBytes + kk * 32),
                                             sdesc_at(dk, (PAGED ? sub * 1024 : sub * (kSubBytes / 2)) + kk * 32), idS,
                                             (c | sub | kk) ? 1u : 0u);
                    } else {
                        const uint64_t dq = sdesc_at(dQk, C::kSubs * c * kSubBytes);
                        const uint64_t dk = PAGED ? sdesc_sw128(kslot, 16, C::kPagedGroupStride) : sdesc_sw128(kslot, 16, 1024);
#pragma unroll
                        for (int sub = 0; sub < C::kSubs; ++sub)
#pragma unroll
                            for (int kk = 0; kk < 4; ++kk) {
                                const uint64_t ad = sdesc_at(dq, sub * kSubBytes + kk * 32);
                                const uint64_t bd = sdesc_at(dk, (PAGED ? sub * 1024 : sub * kSubBytes) + kk * 32);
                                umma_bf16_ss(dst, ad, bd, idS, (c | sub | kk) ? 1u : 0u);
                            }
                    }
                    release_slot();
                }
                commit(&s_full[buf]);
                return true;
            };
            auto issue_pv = [&](int j) -> bool {
                for (int c = 0; c < C::kVChunks; ++c) {
                    if (!next_slot()) return false;
                    if (tail_fix && j == n - 1 && c == 0) {  // the producer zeroed the rows past the end
                        if (!mbar_wait(smem_u32(vfix), 0, abort_flag, a.status, 0x1f)) return false;
                        tc_fence_after();
                    }
                    const uint32_t vslot = sSlots + slot * C::kSlotBytes;
                    // P of step j, packed bf16 pairs: keys 64 hf .. 64 hf + 63 at columns 64 hf .. 64 hf + 31
                    const uint32_t tP = tS0 + (j % C::kSBuf) * 128;
                    const uint64_t dv = PAGED ? sdesc_sw128(vslot, 1024, C::kPagedGroupStride) : sdesc_sw128(vslot, kSubBytes, 1024);
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk) {  // 16 keys per step
                        const uint64_t bd = sdesc_at(dv, PAGED ? kk * 2 * C::kPagedGroupStride : kk * 2048);
                        if (PAIR)
                            umma_pair_ts(tO, tP + (kk >> 2) * 64 + (kk & 3) * 8, bd, idO, (j > 0 || kk > 0) ? 1u : 0u);
                        else
                            umma_bf16_ts(tO + c * C::kSlotCols, tP + (kk >> 2) * 64 + (kk & 3) * 8, bd, idO,
                                         (j > 0 || kk > 0) ? 1u : 0u);
                    }
                    release_slot();
                }
                commit(&pv_done[j % C::kSBuf]);
                return true;
            };
            for (int b = 0; ok && b < C::kSBuf && b < n; ++b) ok = issue_s(b);
            for (int j = 0; ok && j < n; ++j) {
                ok = mbar_wait(smem_u32(&p_full[j % C::kSBuf]), (j / C::kSBuf) & 1, abort_flag, a.status, 0x14);
                if (!ok) break;
                tc_fence_after();
                ok = issue_pv(j);
                // S(j + kSBuf) over the buffer P(j) came from: the pipe runs in order, so P V(j)
                // has read P(j) first
                if (ok && j + C::kSBuf < n) ok = issue_s(j % C::kSBuf);
            }
            // every issued UMMA has finished before TMEM may be released
            if (PAIR) umma_commit_pair(smem_u32(mma_idle), (uint16_t)1);
            else umma_commit(smem_u32(mma_idle));
            mbar_drain(smem_u32(mma_idle), 0, a.status, 0x1a);
        }
    } else {
        // --------------------------------- softmax --------------------------------------
        // Warps w and w + 4 share TMEM lane quarter w & 3 (query rows 32 (w & 3) ..); warp half
        // hf takes the step's score columns (keys) 64 hf .. 64 hf + 63 and the O columns
        // kDV/2 hf .. kDV/2 hf + kDV/2 - 1 of every rescale and of the epilogue. The pair
        // exchanges its row maxima through shared memory every step (named barrier 1 + quarter,
        // 64 threads) and its row sums once at the end. Every exit decision is taken jointly
        // (bar.red.and), so neither warp leaves its partner waiting at a barrier.
        const int quad = warp & 3;
        const int hf = (warp - 2) >> 2;
        const int r = quad * 32 + lane;  // query row within the tile == TMEM lane
        const int qi = qp0 + r;          // position of the query in its sequence
        const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
        const uint32_t pair_bar = 1 + quad;
        float* xch = reinterpret_cast<float*>(smem + C::kOffXch);  // [2][128]
        float m_ref = -INFINITY, l = 0.f;
        bool ok = true;
        for (int j = 0; j < n; ++j) {
            const int buf = j % C::kSBuf;
            bool okw = __all_sync(0xffffffffu,
                                  mbar_wait(smem_u32(&s_full[buf]), (j / C::kSBuf) & 1, abort_flag, a.status, 0x15));
            float s[64];
            float mx = -INFINITY;
            if (okw) {
                tc_fence_after();
                {
                    uint32_t raw[2][32];
#pragma unroll
                    for (int c = 0; c < 2; ++c) tmem_ld32(tS0 + buf * 128 + 64 * hf + c * 32 + lane_base, raw[c]);
                    tmem_ld_wait();
#pragma unroll
                    for (int c = 0; c < 2; ++c)
#pragma unroll
                        for (int e = 0; e < 32; ++e) s[c * 32 + e] = __uint_as_float(raw[c][e]);
                }
                const int key0 = (t_begin + j) * kBKV + 64 * hf;
                const bool edge = (key0 + 63 > qp0) || (a.window > 0 && qp0 + kBQ - 1 - key0 >= a.window) ||
                                  (key0 + 64 > L);
                if (edge) {
#pragma unroll
                    for (int c = 0; c < 64; ++c) {
                        const int key = key0 + c;
                        const bool allowed = key <= qi && key < L && (a.window <= 0 || qi - key < a.window);
                        if (!allowed) s[c] = -INFINITY;
                    }
                }
                // this half's row max over eight independent partials
                float m8[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) m8[i] = s[i];
#pragma unroll
                for (int c = 8; c < 64; c += 8)
#pragma unroll
                    for (int i = 0; i < 8; ++i) m8[i] = fmaxf(m8[i], s[c + i]);
                mx = fmaxf(fmaxf(fmaxf(m8[0], m8[1]), fmaxf(m8[2], m8[3])),
                           fmaxf(fmaxf(m8[4], m8[5]), fmaxf(m8[6], m8[7])));
                xch[hf * 128 + r] = mx;
            }
            ok = named_bar_and(pair_bar, 64, okw);
            if (!ok) break;
            mx = fmaxf(mx, xch[(1 - hf) * 128 + r]);  // the row's max over all 128 keys
            named_bar_sync(pair_bar, 64);             // both read before the buffer is reused
            const float m_tile = mx * a.scale_log2;   // -inf stays -inf (scale > 0)
            float alpha = 1.f;
            const bool moved = m_tile > m_ref + kRescaleLog2;
            if (moved) {
                alpha = m_ref == -INFINITY ? 0.f : fast_exp2(m_ref - m_tile);
                m_ref = m_tile;
            }
            const float m_use = m_ref == -INFINITY ? 0.f : m_ref;
            float rs[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
            uint32_t pk[32];
#pragma unroll
            for (int c = 0; c < 64; c += 2) {
                const float p0 = fast_exp2(fmaf(s[c], a.scale_log2, -m_use));
                const float p1 = fast_exp2(fmaf(s[c + 1], a.scale_log2, -m_use));
                rs[(c >> 1) & 7] += p0 + p1;
                pk[c >> 1] = pack_bf16x2(p0, p1);
            }
            const float rowsum = ((rs[0] + rs[1]) + (rs[2] + rs[3])) + ((rs[4] + rs[5]) + (rs[6] + rs[7]));
            l = l * alpha + rowsum;  // this half's share of the row sum
            // the pair takes the same branches: `moved` depends on the row only
            if (j > 0 && __any_sync(0xffffffffu, moved)) {
                // rescale O: P V(j-1), and so every earlier P V (the MMA pipe completes in order),
                // must be complete. Its barrier has no older phase pending: s_full(j) implies
                // P V(j - kSBuf) is complete.
                const int jp = j - 1;
                okw = __all_sync(0xffffffffu, mbar_wait(smem_u32(&pv_done[jp % C::kSBuf]), (jp / C::kSBuf) & 1,
                                                        abort_flag, a.status, 0x16));
                ok = named_bar_and(pair_bar, 64, okw);
                if (!ok) break;
                tc_fence_after();
                const float f = moved ? alpha : 1.f;
#pragma unroll 1
                for (int c = hf * (C::kDV / 64); c < (hf + 1) * (C::kDV / 64); ++c) {
                    uint32_t raw[32];
                    tmem_ld32(tO + c * 32 + lane_base, raw);
                    tmem_ld_wait();
#pragma unroll
                    for (int e = 0; e < 32; ++e) raw[e] = __float_as_uint(__uint_as_float(raw[e]) * f);
                    tmem_st32(tO + c * 32 + lane_base, raw);
                }
            }
            // P: this half's 64 keys -> the first 32 columns of its half of the step's S buffer
            // (its own scores, already in registers)
            tmem_st32(tS0 + buf * 128 + 64 * hf + lane_base, pk);
            tmem_st_wait();
            tc_fence_before();
            if (PAIR) {  // one arrival per warp, on the even CTA's barrier (it issues P V for both)
                __syncwarp();
                if (lane == 0) {
                    if (crank == 0) mbar_arrive(smem_u32(&p_full[buf]));
                    else mbar_arrive_cluster(lead_bar(&p_full[buf]));
                }
            } else {
                mbar_arrive(smem_u32(&p_full[buf]));
            }
        }
        // ---- epilogue: O / l -> bf16, lse -------------------------------------------------
        // the last P V, and so every earlier one; its barrier has no older phase pending
        bool okw = ok;
        if (okw)
            okw = mbar_wait(smem_u32(&pv_done[(n - 1) % C::kSBuf]), ((n - 1) / C::kSBuf) & 1, abort_flag, a.status, 0x17);
        okw = __all_sync(0xffffffffu, okw);
        if (ok) xch[hf * 128 + r] = l;  // the exchange buffer is free: both read it before the last barrier
        ok = named_bar_and(pair_bar, 64, ok && okw);
        tc_fence_after();
        if (ok) {
            l += xch[(1 - hf) * 128 + r];
            const int qrow = q0 + r;  // query row index within the sequence's rows
            const bool row_ok = qrow < nq;
            const bool packed = PAGED || a.cu_seqlens;
            const float inv = l > 0.f ? 1.f / l : 0.f;
            uint16_t* orow = a.o + ((size_t)(packed ? seq_start + qrow : seq * a.S + qrow) * a.Hq + h) * a.D + dv0;
#pragma unroll 1
            for (int c = hf * (C::kDV / 64); c < (hf + 1) * (C::kDV / 64); ++c) {
                uint32_t raw[32];
                tmem_ld32(tO + c * 32 + lane_base, raw);
                tmem_ld_wait();
                if (row_ok) {
#pragma unroll
                    for (int e = 0; e < 32; e += 8) {
                        uint4 w;
                        w.x = pack_bf16x2(__uint_as_float(raw[e]) * inv, __uint_as_float(raw[e + 1]) * inv);
                        w.y = pack_bf16x2(__uint_as_float(raw[e + 2]) * inv, __uint_as_float(raw[e + 3]) * inv);
                        w.z = pack_bf16x2(__uint_as_float(raw[e + 4]) * inv, __uint_as_float(raw[e + 5]) * inv);
                        w.w = pack_bf16x2(__uint_as_float(raw[e + 6]) * inv, __uint_as_float(raw[e + 7]) * inv);
                        *reinterpret_cast<uint4*>(orow + c * 32 + e) = w;
                    }
                }
            }
            if (row_ok && split == 0 && hf == 0) {
                const float lse = l > 0.f ? (m_ref + __log2f(l)) * 0.69314718055994531f : -INFINITY;
                const size_t li = packed ? (size_t)h * a.T + seq_start + qrow : ((size_t)seq * a.Hq + h) * a.S + qrow;
                a.lse[li] = lse;
            }
        }
        tc_fence_before();
    }
    __syncthreads();
    if (PAIR) {  // the even CTA has drained every copy and product of the pair
        tc_fence_before();
        cluster_sync_all();
    }
    if (warp == 1) {
        tc_fence_after();
        if (PAIR) tmem_dealloc_pair(tbase, 512);
        else tmem_dealloc(tbase, 512);
    }
    if (PAIR) cluster_sync_all();  // neither CTA leaves while the other may still address it
}

template <int DQK, bool PAGED, bool PAIR>
cudaError_t launch_fwd_t(const FwdLaunch& L, cudaStream_t stream) {
    using C = FwdCfg<DQK, PAIR>;
    FwdArgs a;
    a.o = L.o, a.lse = L.lse, a.cu_seqlens = L.cu_seqlens, a.status = L.status;
    a.block_table = L.block_table, a.seq_lens = L.seq_lens, a.cu_q = L.cu_q;
    a.max_pages = L.max_pages, a.num_pages = L.num_pages;
    a.Hq = L.Hq, a.Hkv = L.Hkv, a.S = L.S, a.D = L.D, a.window = L.window;
    a.n_qtiles = (L.S + kBQ - 1) / kBQ;
    a.nsplit = DQK / C::kDV;
    a.T = L.total_rows;
    a.scale_log2 = L.scale * 1.4426950408889634f;
    cudaError_t e =
        cudaFuncSetAttribute(fwd_kernel<DQK, PAGED, PAIR>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::kSmem);
    if (e != cudaSuccess) return e;
    dim3 grid(L.Hq, L.nseq * a.nsplit, a.n_qtiles);
    static const char* const kNames[2][4] = {{"fwd_d64", "fwd_d128", "fwd_d256", "fwd_d512"},
                                             {"fwd_paged_d64", "fwd_paged_d128", "fwd_paged_d256", "fwd_paged_d512"}};
    const char* name = kNames[PAGED ? 1 : 0][DQK == 64 ? 0 : DQK == 128 ? 1 : DQK == 256 ? 2 : 3];
    const ProfMark m = prof_begin(stream, name);
    if (PAIR) {
        // CTA pairs along the head dimension: query heads 2i, 2i + 1 (one GQA group) share the keys
        cudaLaunchConfig_t cfg = {};
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 2;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.gridDim = grid;
        cfg.blockDim = dim3(kThreads);
        cfg.dynamicSmemBytes = C::kSmem;
        cfg.stream = stream;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        e = cudaLaunchKernelEx(&cfg, fwd_kernel<DQK, PAGED, PAIR>, L.tq, L.tk_half, L.tv, a);
        prof_end(stream, m);
        if (e != cudaSuccess) return e;
        return cudaGetLastError();
    }
    fwd_kernel<DQK, PAGED, PAIR><<<grid, kThreads, C::kSmem, stream>>>(L.tq, L.tk, L.tv, a);
    prof_end(stream, m);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd(const FwdLaunch& L, cudaStream_t stream) {
    if (L.nseq == 0 || L.S == 0) return cudaSuccess;
    const bool paged = L.block_table != nullptr;
    // CTA pairs when two consecutive query heads always share a KV head (an even GQA group), at
    // head_dim 512: there each CTA streams 192 KB of keys and values per key step alone, against
    // 96 KB in a pair. At head_dim 256 the sliding-window workload (about nine key steps per
    // CTA) measured slower in pairs (0.713 against 0.665 ms), the pair's fixed cost outweighing
    // the halved stream, so 256 keeps single CTAs.
    const bool pair = L.pair_ok && (L.Hq / L.Hkv) % 2 == 0 && L.D == 512;
    if (L.D == 64) return paged ? launch_fwd_t<64, true, false>(L, stream) : launch_fwd_t<64, false, false>(L, stream);
    if (L.D == 128) return paged ? launch_fwd_t<128, true, false>(L, stream) : launch_fwd_t<128, false, false>(L, stream);
    if (L.D == 256)
        return paged ? launch_fwd_t<256, true, false>(L, stream)
                     : pair ? launch_fwd_t<256, false, true>(L, stream) : launch_fwd_t<256, false, false>(L, stream);
    if (L.D == 512)
        return paged ? (pair ? launch_fwd_t<512, true, true>(L, stream) : launch_fwd_t<512, true, false>(L, stream))
                     : pair ? launch_fwd_t<512, false, true>(L, stream) : launch_fwd_t<512, false, false>(L, stream);
    return cudaErrorInvalidValue;
}

}  // namespace attn
