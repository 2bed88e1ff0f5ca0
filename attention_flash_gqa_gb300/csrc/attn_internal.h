// Internal launch interfaces between the host API (api.cu) and the kernel files.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace attn {

// ---- launch accounting (api.cu) ------------------------------------------------------------
// Every kernel launch of the library goes through these: a process-wide launch counter and,
// when profiling is on, a CUDA event pair on the launching stream.
struct ProfMark {
    int slot = -1;
};
ProfMark prof_begin(cudaStream_t stream, const char* kernel);
void prof_end(cudaStream_t stream, ProfMark m);

// ---- paged decode -----------------------------------------------------------------------
// tk / tv: 3-D maps over the caches (D, Hkv, num_pages * 16) with a D x hb x 16 box, no swizzle;
// used only when the KV heads are split into several blocks (hb < Hkv).
struct DecodeLaunch {
    CUtensorMap tk, tv;
    const uint16_t *q, *k_cache, *v_cache;
    const int32_t *block_table, *seq_lens;
    uint16_t* o;
    float* lse;
    float* part;
    unsigned* status;
    int B, Hq, Hkv, D, max_pages, num_pages, grid, window;
    float scale;
};
size_t decode_smem_bytes(int hb, int D);
int decode_max_grid();
int decode_row_floats(int D);              // floats per (slot, head) partial row
int decode_heads_per_unit(int Hkv, int D, int G);  // hb: KV heads per unit (divides Hkv)
bool decode_packed_layout(int G, int D);  // K, V copied as [64-dim half][head][token][64], 128-byte swizzled
cudaError_t launch_decode_paged(const DecodeLaunch& L, cudaStream_t stream);

// ---- prefill forward ---------------------------------------------------------------------
// q/k/v tensor maps are 4-D over [D, H, S, B] (varlen: B = 1, S = total tokens) with a
// 64 x 1 x 128 x 1 box and 128-byte swizzle. Paged prefill: q as varlen over the packed new
// tokens; k/v over the caches as 5-D (64, 8, Hkv*D/64, 2, num_pages) with a 64 x 8 x 2 x 2 x 1
// box (16 rows x 128 dims of one head of one page).
struct FwdLaunch {
    CUtensorMap tq, tk, tv;
    CUtensorMap tk_half;        // k with a 64 x 1 x 64 x 1 box (CTA-pair forward: half a key tile per CTA)
    bool pair_ok = false;       // tk_half is valid: the CTA-pair forward may be used
    uint16_t* o;
    float* lse;
    const int32_t* cu_seqlens;  // null: dense (or paged)
    unsigned* status;
    int nseq;                   // B (dense), num_seqs (varlen) or num_reqs (paged)
    int Hq, Hkv, S, D;          // S: dense sequence length, max_seqlen (varlen) or max new tokens (paged)
    int total_rows;             // B*S (dense), total tokens (varlen) or total new tokens (paged)
    int window;
    float scale;
    // paged prefill (block_table non-null): request b's n_b = cu_q[b+1] - cu_q[b] new tokens
    // are the last n_b of its seq_lens[b] cached tokens
    const int32_t* block_table = nullptr;  // [num_reqs, max_pages]
    const int32_t* seq_lens = nullptr;
    const int32_t* cu_q = nullptr;
    int max_pages = 0, num_pages = 0;
};
cudaError_t launch_fwd(const FwdLaunch& L, cudaStream_t stream);

// ---- backward ---------------------------------------------------------------------------
struct BwdLaunch {
    CUtensorMap tq, tk, tv, tdo;
    CUtensorMap tqh, tdoh;  // q / dO with a 64 x 1 x (256*128/D) x 1 box: one cluster CTA's query share
    CUtensorMap tdq;  // fp32 dQ accumulator, 4-D [D, Hq, S, B], box 32 x 1 x 128 x 1, 128-byte swizzle
    const uint16_t *q, *k, *v, *o, *dO;
    const float* lse;
    uint16_t *dQ, *dK, *dV;
    float* dq_acc;  // [rows, Hq, D] fp32
    float* delta;   // same layout as lse
    const int32_t* cu_seqlens;
    unsigned* status;
    int nseq, Hq, Hkv, S, D, total_rows, window;
    float scale;
};
cudaError_t launch_bwd(const BwdLaunch& L, cudaStream_t stream);
// main kernel of the backward at D = 64 / 128 (one CTA per key tile; attn_bwd_small.cu)
template <int D>
cudaError_t launch_bwd_small_main(const BwdLaunch& L, cudaStream_t stream);

// ---- merge of attention results over disjoint key sets -----------------------------------
struct MergeLaunch {
    const uint16_t* o_parts;  // [P, B, S, H, D] bf16
    const float* lse_parts;   // [P, B, H, S]
    uint16_t* o;              // [B, S, H, D]
    float* lse;               // [B, H, S]
    int P, B, S, H, D;        // D in {64, 128, 256, 512}
    int sms;
};
cudaError_t launch_merge_lse(const MergeLaunch& L, cudaStream_t stream);

}  // namespace attn
