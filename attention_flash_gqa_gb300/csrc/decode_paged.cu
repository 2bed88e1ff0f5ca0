// Single-token decode over a paged KV cache (D = 128 or 256, page = 16 tokens), optionally
// restricted to a sliding window.
//
// Source: "flex_attention + paged KV + CUDA graphs vs vLLM", sections "What each
// option did" (page-table indirection per block, contiguous blocks, more warps) and
// "Architecture notes" (PagedKVCache + PageTable); "What broke correctness" (a row
// whose mask has no allowed key must not produce NaN). The window: the head_dim 256
// sliding-window layers of "Gemma4 FFPA attention backend support ..." (opening summary)
// at inference, the query at position L-1 seeing keys max(0, L-W) .. L-1.
//
// Design (memory bound: every cached K/V byte in the window is read exactly once):
//  * A unit is one page (16 tokens) of a block of hb KV heads, 32 KB of K and 32 KB of V
//    at most (hb = 8 heads at D = 128, 4 at D = 256). When the block is every head the
//    page is contiguous and K and V are fetched with two untiled TMA bulk copies; otherwise
//    with two 3-D tensor copies (16 tokens x hb heads x D) into a 3-stage ring. In the packed
//    layout below V is always one 5-D tensor copy with the 128-byte swizzle. KV-head
//    blocks are the grid's y dimension; each block runs the scheme below on its heads.
//  * With a window only the pages that hold keys of the window are units; tokens of the
//    window's first page below L-W are masked like the slots past L in the last page.
//  * Work is balanced by pages, not by requests: the pages of all requests are laid
//    end to end and CTA k takes the k-th equal share. A CTA may cover the tail of one
//    request and the head of the next.
//  * Consumer warps serve one KV head each (two per head on the two halves of the page's
//    tokens when a warp's registers cannot hold the whole head): each serves all query heads
//    of the head's GQA group (one K/V row read feeds all of them) with its own running
//    softmax state. D = 128 (GQA groups up to 8): one warp per head; S = Q K^T and
//    O += P V over the page are warp-level MMAs with the group's heads as rows, over K and V
//    copied swizzled, and the softmax stays in registers (see the consumer). D = 256: two
//    warps per head, lane l owns dims 8l..8l+7 with fp32 FMAs, and per-token dot products are
//    finished by a butterfly reduce-scatter across the lanes that split a token.
//  * fp32 online softmax in the log2 domain. Every (CTA, token half) touching a request
//    leaves unnormalised partials (o, m, l) in the workspace, with no wait of any kind, and
//    streams on. A second, small kernel merges each request's partials once the decode grid
//    has finished: it is launched with programmatic stream serialisation, so it is resident
//    before that and its launch costs nothing on the critical path. (A first version had the
//    last CTA to finish a request merge it in-kernel, behind an arrival counter: CTAs whose
//    range ended a request mid-stream stalled for the write-back, the atomic and the merge,
//    and finished the grid late.)
#include <cuda_runtime.h>

#include "attn_internal.h"
#include "ptx.cuh"

namespace attn {
namespace {

constexpr int kPage = 16;
constexpr int kStages = 3;
constexpr int kMaxConsumerWarps = 16;
constexpr int kUnitBytes = 32768;  // K (or V) bytes of one unit at most: 16 tokens x hb heads x D
// D = 128 uses one consumer warp per KV head, whose products are warp MMAs over the whole page;
// D = 256 uses two warps per head (fp32 FMAs, the query and output dims of every head in
// registers). Every configuration runs 8 consumer warps.
template <int G, int D>
struct DecCfg {
    static constexpr bool PACKED = D == 128 && G <= 8;  // decode_packed_layout(G, D): warp MMAs
    // the fp32-FMA layout (head_dim 256): dims per lane, and lanes that split one token's dims
    static constexpr int QD = 8;
    static constexpr int NL = 32;
    static constexpr int WPH = PACKED ? 1 : 2;             // consumer warps per KV head
    // KV heads per unit at most: 32 KB of K per stage
    static constexpr int HB = kUnitBytes / (kPage * D * 2);
    static constexpr int CW = WPH * HB;                    // consumer warps
    static constexpr int TPW = 16 / WPH;                   // page tokens per warp
    // A producer warp of its own, or (packed) none: see the kernel
    static constexpr bool OWN_PRODUCER = !PACKED;
    static constexpr int kThreads = (CW + (OWN_PRODUCER ? 1 : 0)) * 32;
    static constexpr int kRowF = D + 4;  // partial row: o[D], m, l, 2 pad floats (float4 alignment)
    static_assert(PACKED || QD * NL == D, "lanes x dims per lane must cover the head");
    static_assert(CW <= kMaxConsumerWarps, "consumer warps");
};
constexpr int kMaxB = 4096;
constexpr int kMaxUnits = 2048;  // page-table entries of a CTA's range staged in shared memory

struct DecodeArgs {
    const uint16_t* q;
    const uint16_t* kc;
    const uint16_t* vc;
    const int32_t* block_table;
    const int32_t* seq_lens;
    uint16_t* o;
    float* lse;
    float* part;       // [(B + grid) * 2 slots][Hq][D + 4]
    unsigned* status;
    int B, Hq, Hkv, max_pages, num_pages;
    int window;        // <= 0: none
    int hb, nhb;       // KV heads per unit, head blocks (hb * nhb = Hkv)
    float scale_log2;
};

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// d += a b on one warp: a 16 x 16 (row-major), b 16 x 8 (column-major), bf16 in, fp32 out.
// Fragments: g = lane / 4, c = lane % 4; a = {(g, 2c..2c+1), (g+8, 2c..), (g, 2c+8..), (g+8, 2c+8..)},
// b = {(2c..2c+1, g), (2c+8.., g)}, d = {(g, 2c), (g, 2c+1), (g+8, 2c), (g+8, 2c+1)}.
__device__ __forceinline__ void mma_16x8x16_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                                 uint32_t b0, uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Four 8 x 8 b16 matrices from shared memory: lanes 8i .. 8i+7 give the row addresses of matrix i;
// lane (g, c) receives columns 2c, 2c+1 of row g of each.
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}
// The same, transposed: lane (g, c) receives rows 2c, 2c+1 of column g of each.
__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

// Clamped length of request b (records a bounds fault for lengths beyond the table).
__device__ __forceinline__ int req_len(const DecodeArgs& a, int b) {
    int L = a.seq_lens[b];
    int cap = a.max_pages * kPage;
    if (L < 0 || L > cap) {
        atomicOr(a.status, DEVSTAT_BOUNDS);
        L = L < 0 ? 0 : cap;
    }
    return L;
}

// First token the query of a request of length L sees (the window's start).
__device__ __forceinline__ int first_token(const DecodeArgs& a, int L) {
    return a.window > 0 && L > a.window ? L - a.window : 0;
}

// Units (pages holding keys the query sees) of a request of length L.
__device__ __forceinline__ int req_units(const DecodeArgs& a, int L) {
    return L > 0 ? (L - 1) / kPage - first_token(a, L) / kPage + 1 : 0;
}

// CTA that owns global page unit u when P units are split evenly over G CTAs
// (CTA k owns [floor(kP/G), floor((k+1)P/G))).
__device__ __forceinline__ int owner_of(long long u, long long P, int G) {
    return (int)(((u + 1) * (long long)G - 1) / P);
}

template <int G, int D>
__global__ void __launch_bounds__(DecCfg<G, D>::kThreads, 1)
    decode_paged_kernel(const __grid_constant__ CUtensorMap tk, const __grid_constant__ CUtensorMap tv, DecodeArgs a) {
    using DC = DecCfg<G, D>;
    constexpr int kThreads = DC::kThreads;
    constexpr int kConsumerWarps = DC::CW;
    constexpr int kRowF = DC::kRowF;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int hbk = blockIdx.y;         // head block
    const int g0 = hbk * a.hb;          // its first KV head
    const int page_bytes = kPage * a.hb * D * 2;
    uint8_t* stage_base = smem;  // kStages x (K page, V page)
    int32_t* start = reinterpret_cast<int32_t*>(smem + kStages * 2 * page_bytes);  // [B + 1]
    float* scratch = reinterpret_cast<float*>(start + kMaxB + 8);                  // per warp: sc[8G], sp[8G]
    uint64_t* bars = reinterpret_cast<uint64_t*>(scratch + kMaxConsumerWarps * 16 * 8);
    uint64_t* full = bars;
    uint64_t* empty = bars + kStages;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + 2 * kStages);
    int* warp_sums = const_cast<int*>(abort_flag) + 2;  // [8]
    int* released = warp_sums + 8;                       // [kStages] consumer warps done with a stage
    int32_t* unit_tab = reinterpret_cast<int32_t*>(reinterpret_cast<uint8_t*>(bars) + 256);  // [kMaxUnits]

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int B = a.B;
    // Launched with programmatic stream serialisation, so the grid may start while the kernel
    // before it on the stream still runs when that kernel allows it (the merge kernel of a previous
    // decode call does; a kernel launched without the attribute finishes first). The prologue
    // and the first page copies read only seq_lens, block_table and the caches; the consumer
    // warps wait (griddepcontrol.wait) for the predecessor's completion before they read q or
    // write the partials, so the call keeps plain stream order for everything else. The merge
    // kernel that follows may be scheduled at once: it waits for this grid before it reads.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(smem_u32(&full[s]), 1);
            mbar_init(smem_u32(&empty[s]), kConsumerWarps);
        }
        *abort_flag = 0;
        for (int s = 0; s < kStages; ++s) released[s] = 0;
        fence_mbar_init();
    }

    // ---- page prefix sums over requests: start[b] = pages before request b ----------
    {
        const int per = (B + 255) / 256;
        int local = 0;
        if (tid < 256) {
            for (int i = 0; i < per; ++i) {
                int b = tid * per + i;
                if (b < B) local += req_units(a, req_len(a, b));
            }
        }
        // inclusive scan of `local` over threads 0..255
        int v = local;
        for (int off = 1; off < 32; off <<= 1) {
            int n = __shfl_up_sync(0xffffffffu, v, off);
            if (lane >= off) v += n;
        }
        if (tid < 256 && lane == 31) warp_sums[warp] = v;
        __syncthreads();
        int before = 0;
        if (tid < 256)
            for (int w = 0; w < warp; ++w) before += warp_sums[w];
        int excl = before + v - local;
        if (tid < 256) {
            int acc = excl;
            for (int i = 0; i < per; ++i) {
                int b = tid * per + i;
                if (b < B) {
                    start[b] = acc;
                    acc += req_units(a, req_len(a, b));
                }
            }
            if (tid == 255) start[B] = acc;
        }
        __syncthreads();
    }
    const long long P = start[B];
    // Pages are shared by Gc = min(grid, P) CTAs, so every participating CTA owns at
    // least one page and the CTAs touching a request are exactly owner(first)..owner(last).
    const int Gc = (int)(P < (long long)gridDim.x ? P : (long long)gridDim.x);
    const int k = blockIdx.x;

    if (P == 0 || k >= Gc) return;
    const long long u0 = (long long)k * P / Gc, u1 = (long long)(k + 1) * P / Gc;
    if (u0 >= u1) return;

    // first request overlapping [u0, u1): largest b with start[b] <= u0 and a nonempty range
    int b_first = 0;
    {
        int lo = 0, hi = B - 1;
        while (lo < hi) {
            int mid = (lo + hi + 1) >> 1;
            if (start[mid] <= u0) lo = mid;
            else hi = mid - 1;
        }
        b_first = lo;
        while (b_first < B && start[b_first + 1] <= u0) ++b_first;
    }

    // (No L2 prefetch of the later requests' query rows here: it made graph-replayed calls
    // 0.35 us slower.)
    // Page table of this CTA's range, gathered once by all threads: entry = page id << 5 |
    // valid tokens in the page (1..16), or -1 for a page id outside the pool. The loops below
    // then never wait on a dependent global load.
    const int n_units = (int)(u1 - u0);
    auto make_entry = [&](int kk) -> int32_t {
        const long long u = u0 + kk;
        int lo = b_first, hi = B - 1;
        while (lo < hi) {
            int mid = (lo + hi + 1) >> 1;
            if (start[mid] <= u) lo = mid;
            else hi = mid - 1;
        }
        const int L = req_len(a, lo);
        const int p = (int)(u - start[lo]) + first_token(a, L) / kPage;  // page index in the request
        const int page = a.block_table[(size_t)lo * a.max_pages + p];
        if (page < 0 || page >= a.num_pages) {
            atomicOr(a.status, DEVSTAT_BOUNDS);
            return -1;
        }
        const int nt = min(kPage, L - p * kPage);
        return (page << 5) | nt;
    };
    // Warp 0 stages the first units itself and issues their pages at once, so the copies are in
    // flight while the rest of the table is staged.
    const int n_pre = min(n_units, kStages);
    // every cached byte is read once per step: evict-first keeps the stream from displacing
    // (or forcing the write-back of) other lines in L2
    const uint64_t policy = l2_policy_evict_first();
    auto issue = [&](int i, int32_t entry) {
        const int s = i % kStages;
        const uint32_t fb = smem_u32(&full[s]);
        if (entry >= 0) {
            mbar_expect_tx(fb, 2u * page_bytes);
            const uint32_t dk = smem_u32(stage_base + (size_t)s * 2 * page_bytes), dv = dk + page_bytes;
            if constexpr (DC::PACKED) {
                // K and V as [64-dim half][head][token][64 dims], 128-byte swizzled (the 16-byte
                // chunk c of token t's row at chunk c ^ (t % 8)), for the consumers' matrix loads
                tma_load_5d_hint(dk, &tk, fb, 0, 0, g0, 0, entry >> 5, policy);
                tma_load_5d_hint(dv, &tv, fb, 0, 0, g0, 0, entry >> 5, policy);
            } else if (a.nhb == 1) {  // every head: the page is contiguous
                const size_t off = (size_t)(entry >> 5) * kPage * a.Hkv * D;
                bulk_load_hint(dk, a.kc + off, page_bytes, fb, policy);
                bulk_load_hint(dv, a.vc + off, page_bytes, fb, policy);
            } else {  // 16 tokens x hb heads x D of the page
                tma_load_3d_hint(dk, &tk, fb, 0, g0, (entry >> 5) * kPage, policy);
                tma_load_3d_hint(dv, &tv, fb, 0, g0, (entry >> 5) * kPage, policy);
            }
        } else {
            mbar_arrive(fb);
        }
    };
    // The warp that issues the first pages (the producer warp, or consumer warp 0 without one)
    // stages units 0..31 itself
    constexpr int kFirstWarp = DC::OWN_PRODUCER ? kConsumerWarps : 0;
    const int rot = (tid + kThreads - kFirstWarp * 32) % kThreads;
    for (int kk = rot; kk < n_units && kk < kMaxUnits; kk += kThreads) unit_tab[kk] = make_entry(kk);
    if (warp == kFirstWarp) {
        __syncwarp();
        if (lane == 0)
            for (int i = 0; i < n_pre; ++i) issue(i, unit_tab[i]);
    }
    __syncthreads();
    auto unit_entry = [&](int kk) -> int32_t { return kk < kMaxUnits ? unit_tab[kk] : make_entry(kk); };

    if constexpr (DC::OWN_PRODUCER) {
        if (warp == kConsumerWarps) {
            // -------------------------- producer ----------------------------------------
            if (lane == 0) {
                int i = 0;
                for (long long u = u0; u < u1; ++u, ++i) {
                    if (i < n_pre) continue;  // issued before the table was staged
                    const int s = i % kStages, r = i / kStages;
                    if (r > 0 && !mbar_wait(smem_u32(&empty[s]), (r - 1) & 1, abort_flag, a.status, 0x31)) break;
                    issue(i, unit_entry(i));
                }
                // Drain: every issued copy completes before this CTA may exit.
                const int issued = i;
                for (int s = 0; s < kStages && s < issued; ++s) {
                    const int last = s + ((issued - 1 - s) / kStages) * kStages;
                    mbar_drain(smem_u32(&full[s]), (last / kStages) & 1, a.status, 0x33);
                }
            }
            return;
        }
    }
    // Without a producer warp (the packed layout), the consumer warp that releases a stage last
    // refills it with the unit kStages further on; its wait on the stage's empty barrier, which
    // every consumer warp arrives on after its reads, orders those reads before the copy. Eight
    // warps alone put two on each SM scheduler, so a warp may use up to 255 registers; a ninth
    // warp puts three on one scheduler and caps every warp at 168, where the packed consumer
    // spills. Measured at the head_dim 128 decode workload: 35.7 against 36.4 us per call. The
    // other layouts keep their producer warp: the window workload at head_dim 256 took 163.2
    // against 158.4 us without it.
    auto release = [&](int i) -> bool {  // consumer warp done with unit i's stage (lane 0)
        const int s = i % kStages;
        mbar_arrive(smem_u32(&empty[s]));
        if constexpr (DC::OWN_PRODUCER) return true;
        if (atomicAdd(&released[s], 1) != kConsumerWarps - 1) return true;
        released[s] = 0;
        const int inext = i + kStages;
        if (inext >= n_units) return true;
        if (!mbar_wait(smem_u32(&empty[s]), (i / kStages) & 1, abort_flag, a.status, 0x31)) return false;
        issue(inext, unit_entry(inext));
        return true;
    };

    // ---------------------------------- consumers ----------------------------------------
    asm volatile("griddepcontrol.wait;" ::: "memory");
    // Every consumer warp serves one KV head for all G query heads of its group (one K/V
    // row read feeds all of them) with its own running softmax state; when two warps share
    // a head (token halves), they are merged like split partials at the end.
    //  * D = 128 ("packed" layout, one warp per KV head, all 16 tokens of a page): Q K^T and
    //    P V are warp MMAs (below); the o accumulator is O in MMA fragments.
    //  * D = 256 (two warps per KV head, 8 tokens each): lane l owns dims 8l .. 8l+7 of the
    //    warp's 8 tokens (32-lane butterfly).
    constexpr bool PACKED = DC::PACKED;
    constexpr int TPW = DC::TPW;
    const int gl = warp / DC::WPH, half = warp % DC::WPH;  // KV head within the block, token half
    const int g = g0 + gl;                                  // KV head
    const bool active = gl < a.hb;
    float* sc = scratch + warp * 2 * TPW * G;  // [TPW * G] scores (log2 domain), index token * G + head
    float* sp = sc + TPW * G;                  // [TPW * G] probabilities
    constexpr int QD = DC::QD;            // dims per lane
    constexpr int NT = 8;                 // tokens per lane group
    constexpr int NL = DC::NL;            // lanes that split one token's dims
    constexpr int NV = TPW * G;           // (token, head) values of the warp's tokens
    constexpr int NVL = NT * G;           // partial values per lane
    constexpr int NF = NVL >= NL ? NVL / NL : 1;  // finished values per lane after the butterfly
    constexpr int KH = NVL >= NL ? 5 : (NVL == 16 ? 4 : (NVL == 8 ? 3 : (NVL == 4 ? 2 : 1)));
    constexpr int NH = NV >= 32 ? NV / 32 : 1;  // values per lane in the softmax layout
    // (the fp32-FMA layouts)
    const int dim0 = QD * lane;
    const int tok0 = TPW * half;  // first page token of this warp's tokens

    float qv[G][QD];  // this lane's query dims, loaded when the request changes
    float acc_o[G][QD];
#pragma unroll
    for (int hh = 0; hh < G; ++hh)
#pragma unroll
        for (int e = 0; e < QD; ++e) qv[hh][e] = 0.f, acc_o[hh][e] = 0.f;
    // Packed layout: per page S = Q K^T and O += P V are warp MMAs (m16n8k16, bf16 in, fp32 out)
    // with the group's heads as the 16 rows (rows past G are zero). Lane (mg, mc) holds:
    //  * qa: head mg's query as A fragments, dims 16 s + 2 mc, +1 and 16 s + 8 + 2 mc, +1 of k-step s;
    //  * the scores of head mg for tokens 2 mc, 2 mc + 1, 8 + 2 mc, 9 + 2 mc, which are exactly the
    //    A fragment of P for P V, so the softmax runs in registers;
    //  * oa[n]: head mg's output dims 8 n + 2 mc, +1 (n = 0..15).
    // m_run and l_run then belong to head mg (l_run: this lane's share of its 16 tokens).
    const int mg = lane >> 2, mc = lane & 3;
    uint32_t qa[16];
    float oa[16][4];
#pragma unroll
    for (int e = 0; e < 16; ++e) qa[e] = 0u;
#pragma unroll
    for (int n8 = 0; n8 < 16; ++n8)
#pragma unroll
        for (int e = 0; e < 4; ++e) oa[n8][e] = 0.f;
    float m_run = -INFINITY, l_run = 0.f;  // for head lane % G (packed: head mg)

    int b = b_first;
    int i = 0;
    bool ok = true;
    int cur_b = -1;
    int lo_tok = 0;  // first visible token within the request's first unit (window)
    for (long long u = u0; u < u1 && ok; ++u, ++i) {
        while (start[b + 1] <= u) ++b;
        if (b != cur_b) {
            cur_b = b;
            lo_tok = first_token(a, req_len(a, b)) % kPage;
            if (PACKED && active && mg < G) {
                const uint16_t* qrow = a.q + ((size_t)b * a.Hq + g * G + mg) * D + 2 * mc;
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) {
                    qa[2 * ks] = *reinterpret_cast<const uint32_t*>(qrow + 16 * ks);
                    qa[2 * ks + 1] = *reinterpret_cast<const uint32_t*>(qrow + 16 * ks + 8);
                }
            }
            if (!PACKED && active) {  // (the FMA layout)
#pragma unroll
                for (int hh = 0; hh < G; ++hh) {
                    const uint16_t* qrow = a.q + ((size_t)b * a.Hq + g * G + hh) * D + dim0;
                    const uint4 w = *reinterpret_cast<const uint4*>(qrow);
                    const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) qv[hh][2 * e] = bf16_lo(ws[e]), qv[hh][2 * e + 1] = bf16_hi(ws[e]);
                }
            }
        }
        const int s = i % kStages, r = i / kStages;
        ok = mbar_wait(smem_u32(&full[s]), r & 1, abort_flag, a.status, 0x32);
        if (!ok) break;
        const int32_t entry = unit_entry(i);
        const int nt = (entry >= 0 ? (entry & 31) : 0) - TPW * half;  // end of this warp's valid tokens (may be <= 0)
        const int tlo = (u == start[b] ? lo_tok : 0) - TPW * half;     // first of them (may be < 0)
        if (active && nt > 0 && tlo < TPW) {
            const uint8_t* kp = stage_base + (size_t)s * 2 * page_bytes;
            const uint8_t* vp = kp + page_bytes;
            if constexpr (PACKED) {
                const uint32_t kb = smem_u32(kp), vb = smem_u32(vp);
                const uint32_t hbytes = (uint32_t)a.hb * kPage * 128u;  // one 64-dim half of every head
                auto vis = [&](int t) { return t < nt && t >= tlo; };
                // S = Q K^T: tiles of tokens 0-7 and 8-15. Per k-step one matrix load gives both
                // tiles' B fragments: lanes 0-7 / 8-15 / 16-23 / 24-31 address tokens 0-7, 0-7,
                // 8-15, 8-15 at the step's lower / upper / lower / upper 8 dims; the swizzle puts
                // the 8 rows of each matrix in 8 different bank groups.
                float sa[4] = {0.f, 0.f, 0.f, 0.f}, sb[4] = {0.f, 0.f, 0.f, 0.f};
                {
                    const int lt = (lane & 7) + ((lane >> 4) << 3), lhi = (lane >> 3) & 1;
                    const uint32_t krow = kb + (uint32_t)(gl * kPage + lt) * 128u;
#pragma unroll
                    for (int ks = 0; ks < 8; ++ks) {
                        const int ch = 2 * (ks & 3) + lhi;
                        uint32_t k0, k1, k2, k3;
                        ldsm_x4(krow + (ks >> 2) * hbytes + (uint32_t)((ch ^ (lt & 7)) << 4), k0, k1, k2, k3);
                        mma_16x8x16_bf16(sa, qa[2 * ks], 0u, qa[2 * ks + 1], 0u, k0, k1);
                        mma_16x8x16_bf16(sb, qa[2 * ks], 0u, qa[2 * ks + 1], 0u, k2, k3);
                    }
                }
                // head mg, tokens 2 mc, 2 mc + 1, 8 + 2 mc, 9 + 2 mc (log2 units; -inf if not visible)
                const int t0 = 2 * mc;
                float sv[4] = {sa[0], sa[1], sb[0], sb[1]};
                bool over = false;
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int tt = t0 + (e & 1) + 8 * (e >> 1);
                    sv[e] = mg < G && vis(tt) ? sv[e] * a.scale_log2 : -INFINITY;
                    over |= sv[e] > m_run + 8.f;
                }
                // lazy running max, as in the other layouts: it moves only when a score exceeds
                // it by more than 8, so p <= 2^8 and most pages need no rescale
                if (__any_sync(0xffffffffu, over)) {
                    float mx = fmaxf(fmaxf(sv[0], sv[1]), fmaxf(sv[2], sv[3]));
                    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
                    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));  // over head mg's 16 tokens
                    const float m_new = mx > m_run + 8.f ? mx : m_run;
                    const float alpha = m_run == -INFINITY ? 0.f : fast_exp2(m_run - m_new);
                    l_run *= alpha;
#pragma unroll
                    for (int n8 = 0; n8 < 16; ++n8) oa[n8][0] *= alpha, oa[n8][1] *= alpha;
                    m_run = m_new;
                }
                const float m_use = m_run == -INFINITY ? 0.f : m_run;
                float pv[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    pv[e] = sv[e] == -INFINITY ? 0.f : fast_exp2(sv[e] - m_use);
                    l_run += pv[e];
                }
                // O += P V: A = P (bf16, as the prefill's P V takes it), B = V by transposed matrix
                // loads, two 8-dim tiles per load: lanes 0-7 / 8-15 / 16-23 / 24-31 address tokens
                // 0-7, 8-15, 0-7, 8-15 at the lower / lower / upper / upper 8 dims
                const uint32_t pa0 = pack_bf16x2(pv[0], pv[1]), pa1 = pack_bf16x2(pv[2], pv[3]);
                // tokens past the end hold arbitrary bytes: zero them (p is 0 there, but 0 * NaN is not)
                uint32_t vm0 = 0xffffffffu, vm1 = 0xffffffffu;
                if (!(nt >= TPW && tlo <= 0)) {
                    vm0 = (vis(t0) ? 0x0000ffffu : 0u) | (vis(t0 + 1) ? 0xffff0000u : 0u);
                    vm1 = (vis(t0 + 8) ? 0x0000ffffu : 0u) | (vis(t0 + 9) ? 0xffff0000u : 0u);
                }
                {
                    const int lt = (lane & 7) + (((lane >> 3) & 1) << 3), lhi = lane >> 4;
                    const uint32_t vrow = vb + (uint32_t)(gl * kPage + lt) * 128u;
#pragma unroll
                    for (int i8 = 0; i8 < 8; ++i8) {
                        const int ch = 2 * (i8 & 3) + lhi;
                        uint32_t v0, v1, v2, v3;
                        ldsm_x4_trans(vrow + (i8 >> 2) * hbytes + (uint32_t)((ch ^ (lt & 7)) << 4), v0, v1, v2, v3);
                        mma_16x8x16_bf16(oa[2 * i8], pa0, 0u, pa1, 0u, v0 & vm0, v1 & vm1);
                        mma_16x8x16_bf16(oa[2 * i8 + 1], pa0, 0u, pa1, 0u, v2 & vm0, v3 & vm1);
                    }
                }
            } else {
                // partial scores over this lane's dims: v[t * G + hh] for its NT tokens
                float v[NVL];
#pragma unroll
                for (int t = 0; t < NT; ++t) {
                    const uint8_t* krow = kp + ((size_t)((tok0 + t) * a.hb + gl) * D + dim0) * 2;
                    const uint4 w = *reinterpret_cast<const uint4*>(krow);
                    const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
                    float2 k2[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) k2[e] = make_float2(bf16_lo(ws[e]), bf16_hi(ws[e]));
#pragma unroll
                    for (int hh = 0; hh < G; ++hh) {
                        float2 acc = __fmul2_rn(make_float2(qv[hh][0], qv[hh][1]), k2[0]);
#pragma unroll
                        for (int e = 1; e < 4; ++e) acc = __ffma2_rn(make_float2(qv[hh][2 * e], qv[hh][2 * e + 1]), k2[e], acc);
                        v[t * G + hh] = acc.x + acc.y;
                    }
                }
                // butterfly reduce-scatter over the NL lanes of a token group (offsets NL/2 .. 1):
                // after KH halvings a lane holds NF values, index (lane >> (5 - KH)) * NF + j;
                // remaining offsets all-reduce.
                int count = NVL;
#pragma unroll
                for (int off = NL / 2; off >= 1; off >>= 1) {
                    if (count > 1) {
                        const int hf = count >> 1;
                        const bool upper = (lane & off) != 0;
#pragma unroll
                        for (int j = 0; j < NVL / 2; ++j) {
                            if (j < hf) {
                                const float send = upper ? v[j] : v[hf + j];
                                const float keep = upper ? v[hf + j] : v[j];
                                v[j] = keep + __shfl_xor_sync(0xffffffffu, send, off);
                            }
                        }
                        count = hf;
                    } else {
                        v[0] += __shfl_xor_sync(0xffffffffu, v[0], off);
                    }
                }
                if ((lane & ((1 << (5 - KH)) - 1)) == 0) {
#pragma unroll
                    for (int j = 0; j < NF; ++j) {
                        const int idx = (lane >> (5 - KH)) * NF + j;  // t * G + hh within this lane's tokens
                        const int tw = idx / G;                        // token within the warp's 8
                        sc[tw * G + idx % G] = tw < nt && tw >= tlo ? v[j] * a.scale_log2 : -INFINITY;
                    }
                }
                __syncwarp();
                // softmax layout: lane holds idx = lane + 32*j (head lane % G, token idx / G).
                // Lazy running max (as in the prefill forward): m_run, shared by the lanes of a head,
                // moves only when a page's score exceeds it by more than 8 (log2 units), so p <= 2^8
                // and most pages need neither the max reduction nor a rescale of o and l. l_run is
                // this lane's share of the head's sum, reduced across the head's lanes per piece.
                float sv[NH];
                bool over = false;
#pragma unroll
                for (int j = 0; j < NH; ++j) {
                    const int idx = lane + 32 * j;
                    sv[j] = idx < NV ? sc[idx] : -INFINITY;
                    over |= sv[j] > m_run + 8.f;
                }
                if (__any_sync(0xffffffffu, over)) {
                    float mx = -INFINITY;
#pragma unroll
                    for (int j = 0; j < NH; ++j) mx = fmaxf(mx, sv[j]);
#pragma unroll
                    for (int off = G; off < 32; off <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
                    const float m_new = mx > m_run + 8.f ? mx : m_run;
                    // o and l are zero while m_run is -inf
                    const float alpha = m_run == -INFINITY ? 0.f : fast_exp2(m_run - m_new);
                    l_run *= alpha;
#pragma unroll
                    for (int hh = 0; hh < G; ++hh) {
                        const float al = __shfl_sync(0xffffffffu, alpha, hh);
#pragma unroll
                        for (int e = 0; e < QD; ++e) acc_o[hh][e] *= al;
                    }
                    m_run = m_new;
                }
                const float m_use = m_run == -INFINITY ? 0.f : m_run;
#pragma unroll
                for (int j = 0; j < NH; ++j) {
                    const int idx = lane + 32 * j;
                    const float pj = sv[j] == -INFINITY ? 0.f : fast_exp2(sv[j] - m_use);
                    if (idx < NV) sp[idx] = pj;
                    l_run += pj;
                }
                __syncwarp();
                // o update: add this lane's tokens
                const int tmax = nt < 8 ? nt : 8;
                for (int t = tlo > 0 ? tlo : 0; t < tmax; ++t) {  // only the warp's visible tokens
                    const uint8_t* vrow = vp + ((size_t)((TPW * half + t) * a.hb + gl) * D + dim0) * 2;
                    float vv[QD];
                    const uint4 w = *reinterpret_cast<const uint4*>(vrow);
                    const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) vv[2 * e] = bf16_lo(ws[e]), vv[2 * e + 1] = bf16_hi(ws[e]);
#pragma unroll
                    for (int hh = 0; hh < G; ++hh) {
                        const float pt = sp[t * G + hh];
#pragma unroll
                        for (int e = 0; e < QD; ++e) acc_o[hh][e] = fmaf(pt, vv[e], acc_o[hh][e]);
                    }
                }
            }
        }
        __syncwarp();
        bool rel_ok = true;
        if (lane == 0) rel_ok = release(i);
        ok = __shfl_sync(0xffffffffu, rel_ok, 0) && ok;

        // ---- end of this request inside this CTA: write its partials (o, m, l) -----------
        // The merge kernel that follows this grid combines each request's slots.
        if (u + 1 == start[b + 1] || u + 1 == u1) {
            // slot of (request b, CTA k, token half): (b + k) * 2 + half
            float* slot = a.part + ((size_t)(b + k) * 2 + half) * a.Hq * kRowF;
            if (active && PACKED) {
                // head mg's sum: its 4 lanes each hold a share
                l_run += __shfl_xor_sync(0xffffffffu, l_run, 1);
                l_run += __shfl_xor_sync(0xffffffffu, l_run, 2);
                if (mg < G) {
                    float* row = slot + (size_t)(g * G + mg) * kRowF;
#pragma unroll
                    for (int n8 = 0; n8 < 16; ++n8)
                        *reinterpret_cast<float2*>(row + 8 * n8 + 2 * mc) = make_float2(oa[n8][0], oa[n8][1]);
                    if (mc == 0) {
                        row[D] = m_run;
                        row[D + 1] = l_run;
                    }
                }
            } else if (active) {
                // the head's sum: its lanes (lane % G) each hold a share
#pragma unroll
                for (int off = G; off < 32; off <<= 1) l_run += __shfl_xor_sync(0xffffffffu, l_run, off);
#pragma unroll
                for (int hh = 0; hh < G; ++hh) {
                    float* row = slot + (size_t)(g * G + hh) * kRowF;
#pragma unroll
                    for (int e = 0; e < QD; e += 4)
                        *reinterpret_cast<float4*>(row + dim0 + e) =
                            make_float4(acc_o[hh][e], acc_o[hh][e + 1], acc_o[hh][e + 2], acc_o[hh][e + 3]);
                    if (lane == hh) {
                        row[D] = m_run;
                        row[D + 1] = l_run;
                    }
                }
            }
            // reset the running state for the next request
            m_run = -INFINITY, l_run = 0.f;
#pragma unroll
            for (int hh = 0; hh < G; ++hh)
#pragma unroll
                for (int e = 0; e < QD; ++e) acc_o[hh][e] = 0.f;
#pragma unroll
            for (int n8 = 0; n8 < 16; ++n8)
#pragma unroll
                for (int e = 0; e < 4; ++e) oa[n8][e] = 0.f;
        }
    }
    // After a give-up, copies issued into the ring may still be landing: let them finish before
    // the CTA's shared memory is released. (On the normal path every issued copy was waited on.)
    if (!ok) {
        const uint64_t t0 = globaltimer();
        while (globaltimer() - t0 < 100000ull) __nanosleep(1000);
    }
}


// Combines the split partials of every (request, head block): the partial slots of request b are
// those of CTAs kf..kl of the decode grid that covered its units (both token halves when two
// warps share a head). Launched right after the decode kernel with programmatic stream
// serialisation, so its CTAs are resident while the decode grid runs; griddepcontrol.wait
// returns once that grid has finished and its writes are visible. A thread owns one head's 16
// dims and folds the slots in a running maximum, SB slots at a time with all of their loads
// (each slot's m, l and 16 o values) in flight together: a request split over up to SB slots
// is merged in one round trip. A request with no visible key gets o = 0 and lse = -inf.
struct MergeArgs {
    const float* part;
    const int32_t* seq_lens;
    uint16_t* o;
    float* lse;
    unsigned* status;
    int B, Hq, hb, decode_grid, max_pages, window;
};

// Heads of a (request, head block) are split over gridDim.z CTAs of kMergeThreads, one
// 16-dim item per thread, so the merge of a batch runs on every SM.
constexpr int kMergeThreads = 64;

template <int G, int D>
__global__ void __launch_bounds__(kMergeThreads) decode_merge_kernel(MergeArgs m) {
    using DC = DecCfg<G, D>;
    constexpr int kRowF = DC::kRowF;
    constexpr int SB = 8;
    constexpr int DI = 8;  // dims per thread
    // a kernel launched after this one with programmatic serialisation may be scheduled now (it
    // waits for this grid's completion before it reads anything)
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int b = blockIdx.x;
    const int nh = m.hb * G / gridDim.z;  // heads of this CTA
    const int h0 = blockIdx.y * m.hb * G + blockIdx.z * nh;
    // Which decode CTAs covered request b follows from the request lengths alone (inputs, not
    // written by the decode grid): this runs before the wait, beside the decode grid.
    // Every warp sums the unit counts over all requests itself (no shared memory, so these
    // CTAs fit beside a decode CTA).
    DecodeArgs la;  // the fields req_len / req_units read
    la.seq_lens = m.seq_lens, la.max_pages = m.max_pages, la.window = m.window, la.status = m.status;
    long long before = 0, total = 0;
    for (int i = threadIdx.x & 31; i < m.B; i += 32) {
        const int n = req_units(la, req_len(la, i));
        total += n;
        if (i < b) before += n;
    }
#pragma unroll
    for (int off = 16; off; off >>= 1) {
        before += __shfl_xor_sync(0xffffffffu, before, off);
        total += __shfl_xor_sync(0xffffffffu, total, off);
    }
    const long long s0 = before, P = total;
    const long long s1 = s0 + req_units(la, req_len(la, b));
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int Gc = (int)(P < (long long)m.decode_grid ? P : (long long)m.decode_grid);
    const int nitems = nh * (D / DI);
    if (s1 == s0) {
        for (int it = threadIdx.x; it < nitems; it += blockDim.x) {
            const int h = h0 + it / (D / DI), d0 = DI * (it % (D / DI));
            *reinterpret_cast<uint4*>(m.o + ((size_t)b * m.Hq + h) * D + d0) = make_uint4(0, 0, 0, 0);
            if (d0 == 0) m.lse[(size_t)b * m.Hq + h] = -INFINITY;
        }
        return;
    }
    const int kf = owner_of(s0, P, Gc), kl = owner_of(s1 - 1, P, Gc);
    const int nslots = DC::WPH * (kl - kf + 1);
    auto slot_row = [&](int q, int h) -> const float* {
        return m.part + ((size_t)(b + kf + q / DC::WPH) * 2 + q % DC::WPH) * m.Hq * kRowF + (size_t)h * kRowF;
    };
    for (int it = threadIdx.x; it < nitems; it += blockDim.x) {
        const int h = h0 + it / (D / DI), d0 = DI * (it % (D / DI));
        float M = -INFINITY, Ls = 0.f;
        float O[DI];
#pragma unroll
        for (int e = 0; e < DI; ++e) O[e] = 0.f;
        for (int q0 = 0; q0 < nslots; q0 += SB) {
            float2 ml[SB];
            float4 ov[SB][2];
#pragma unroll
            for (int j = 0; j < SB; ++j) {
                ml[j] = make_float2(-INFINITY, 0.f);
                ov[j][0] = ov[j][1] = make_float4(0.f, 0.f, 0.f, 0.f);
                if (q0 + j < nslots) {
                    const float* row = slot_row(q0 + j, h);
                    ml[j] = __ldcg(reinterpret_cast<const float2*>(row + D));
                    ov[j][0] = __ldcg(reinterpret_cast<const float4*>(row + d0));
                    ov[j][1] = __ldcg(reinterpret_cast<const float4*>(row + d0) + 1);
                }
            }
            float Mc = M;
#pragma unroll
            for (int j = 0; j < SB; ++j) Mc = fmaxf(Mc, ml[j].x);
            if (Mc == -INFINITY) continue;
            const float rs = M == -INFINITY ? 0.f : fast_exp2(M - Mc);
            Ls *= rs;
#pragma unroll
            for (int e = 0; e < DI; ++e) O[e] *= rs;
#pragma unroll
            for (int j = 0; j < SB; ++j) {
                const float w = ml[j].x == -INFINITY ? 0.f : fast_exp2(ml[j].x - Mc);  // an empty slot adds nothing
                Ls += w * ml[j].y;
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    O[4 * c] += w * ov[j][c].x, O[4 * c + 1] += w * ov[j][c].y;
                    O[4 * c + 2] += w * ov[j][c].z, O[4 * c + 3] += w * ov[j][c].w;
                }
            }
            M = Mc;
        }
        const float inv = Ls > 0.f ? 1.f / Ls : 0.f;
        uint4 w0;
        w0.x = pack_bf16x2(O[0] * inv, O[1] * inv), w0.y = pack_bf16x2(O[2] * inv, O[3] * inv);
        w0.z = pack_bf16x2(O[4] * inv, O[5] * inv), w0.w = pack_bf16x2(O[6] * inv, O[7] * inv);
        *reinterpret_cast<uint4*>(m.o + ((size_t)b * m.Hq + h) * D + d0) = w0;
        if (d0 == 0) m.lse[(size_t)b * m.Hq + h] = Ls > 0.f ? (M + __log2f(Ls)) * 0.69314718055994531f : -INFINITY;
    }
}

}  // namespace

size_t decode_smem_bytes(int hb, int D) {
    return 1024 + (size_t)kStages * 2 * kPage * hb * D * 2 + (kMaxB + 8) * 4 + (size_t)kMaxConsumerWarps * 16 * 8 * 4 +
           256 + kMaxUnits * 4;
}

int decode_max_grid() { return 256; }
int decode_row_floats(int D) { return D + 4; }

bool decode_packed_layout(int G, int D) { return D == 128 && G <= 8; }

int decode_heads_per_unit(int Hkv, int D, int G) {
    int cap = D > 0 ? (int)(kUnitBytes / (kPage * D * 2)) : 1;
    (void)G;
    if (cap < 1) cap = 1;  // head sizes no decode kernel takes: callers reject them, but never divide by 0
    int hb = Hkv < cap ? Hkv : cap;
    if (hb < 1) hb = 1;
    while (hb > 1 && Hkv % hb) --hb;
    return hb;
}

cudaError_t launch_decode_paged(const DecodeLaunch& L, cudaStream_t stream) {
    DecodeArgs a;
    a.q = L.q, a.kc = L.k_cache, a.vc = L.v_cache, a.block_table = L.block_table, a.seq_lens = L.seq_lens;
    a.o = L.o, a.lse = L.lse, a.part = L.part, a.status = L.status;
    a.B = L.B, a.Hq = L.Hq, a.Hkv = L.Hkv, a.max_pages = L.max_pages, a.num_pages = L.num_pages;
    a.window = L.window;
    const int G = L.Hq / L.Hkv;
    a.hb = decode_heads_per_unit(L.Hkv, L.D, G);
    a.nhb = L.Hkv / a.hb;
    a.scale_log2 = L.scale * 1.4426950408889634f;
    const size_t smem = decode_smem_bytes(a.hb, L.D);
    MergeArgs mg;
    mg.part = L.part, mg.seq_lens = L.seq_lens, mg.o = L.o, mg.lse = L.lse, mg.status = L.status;
    mg.B = L.B, mg.Hq = L.Hq, mg.hb = a.hb, mg.decode_grid = L.grid, mg.max_pages = L.max_pages, mg.window = L.window;
    auto go = [&](auto kern, auto merge, int threads) -> cudaError_t {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        // Both kernels are launched with programmatic stream serialisation: each may be scheduled
        // while its predecessor on the stream still runs, and waits on the device
        // (griddepcontrol.wait) for that predecessor's completion before it reads anything the
        // predecessor may write.
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cudaLaunchConfig_t dcfg = {};
        dcfg.gridDim = dim3(L.grid, a.nhb);
        dcfg.blockDim = dim3(threads);
        dcfg.dynamicSmemBytes = smem;
        dcfg.stream = stream;
        dcfg.attrs = attr;
        dcfg.numAttrs = 1;
        ProfMark m = prof_begin(stream, L.D == 128 ? "decode_paged" : "decode_paged_d256");
        e = cudaLaunchKernelEx(&dcfg, kern, L.tk, L.tv, a);
        prof_end(stream, m);
        if (e != cudaSuccess || (e = cudaGetLastError()) != cudaSuccess) return e;
        cudaLaunchConfig_t cfg = {};
        const int nh = a.hb * G;  // query heads of a head block
        int nz = nh * (L.D / 8) / kMergeThreads;
        if (nz < 1) nz = 1;
        while (nh % nz) --nz;
        cfg.gridDim = dim3(L.B, a.nhb, nz);
        cfg.blockDim = dim3(kMergeThreads);
        cfg.dynamicSmemBytes = 0;
        cfg.stream = stream;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        m = prof_begin(stream, "decode_merge");
        e = cudaLaunchKernelEx(&cfg, merge, mg);
        prof_end(stream, m);
        return e != cudaSuccess ? e : cudaGetLastError();
    };
#define ATTN_DECODE_CASE(G_, D_) \
    case G_: return go(decode_paged_kernel<G_, D_>, decode_merge_kernel<G_, D_>, DecCfg<G_, D_>::kThreads);
    if (L.D == 128) {
        switch (G) {
            ATTN_DECODE_CASE(1, 128)
            ATTN_DECODE_CASE(2, 128)
            ATTN_DECODE_CASE(4, 128)
            ATTN_DECODE_CASE(8, 128)
            default: return cudaErrorInvalidValue;
        }
    }
    if (L.D == 256) {
        switch (G) {
            ATTN_DECODE_CASE(1, 256)
            ATTN_DECODE_CASE(2, 256)
            ATTN_DECODE_CASE(4, 256)
            default: return cudaErrorInvalidValue;
        }
    }
#undef ATTN_DECODE_CASE
    return cudaErrorInvalidValue;
}

}  // namespace attn
