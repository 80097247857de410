// kda_internal.cuh -- declarations shared by the library's translation units
// (host API and kernels).  Not part of the public ABI; see include/kda.h.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace kda {

constexpr int kD = 128;     // Dk = Dv
constexpr int kChunk = 16;  // rows per chunk

// Device status codes (same values as kda_status).
constexpr int32_t kStatusOk = 0;
constexpr int32_t kStatusBadSeqlens = 1;
constexpr int32_t kStatusTimeout = 7;

// Everything a forward launch needs; plain pointers and sizes.
struct FwdParams {
    const __nv_bfloat16* q;
    const __nv_bfloat16* k;
    const __nv_bfloat16* v;
    const float* g;
    const __nv_bfloat16* beta;
    const void* s0;       // [N][H][128][128] fp32 (bf16 when s0_bf16), or nullptr (zero state)
    void* sfin;           // [N][H][128][128] fp32 (bf16 when sfin_bf16), or nullptr (not written)
    __nv_bfloat16* out;   // [T_total][H][128]
    const int32_t* cu;    // [N + 1] or nullptr (dense)
    int64_t T_total;
    int64_t dense_len;    // tokens per sequence when cu == nullptr
    int32_t N;
    int32_t H;            // heads of v, g, beta and the states
    int32_t Hq;           // heads of q (k has min(Hq, H), the output max(Hq, H))
    float scale;
    int64_t wait_limit;   // iteration limit of bounded spin waits
    int32_t debug_flags;  // KDA_DEBUG_* bits (failure-path tests only)
    int32_t* status;      // device status word of this device
    // Segment launches (seg_len > 0).  Dense: CTA row n' = b * nseg_used + s runs segment s
    // of sequence b, tokens [b*L + s*seg_len, b*L + min((s+1)*seg_len, L)), L = dense_len.
    // Varlen (cu != nullptr): row n' is global segment n' of the table seg_start (sequence
    // n owns rows seg_start[n] .. seg_start[n+1]-1, at least one), tokens
    // [cu[n] + s*seg_len, min(cu[n] + (s+1)*seg_len, cu[n+1])); rows past seg_start[N]
    // exit.
    int64_t seg_len;
    int32_t nseg_used;    // dense: segments of each sequence covered by this launch
    int32_t nseg_total;   // dense: segments of each sequence
    int32_t flags;        // kFlag* below
    const int32_t* seg_start;  // varlen segment table [N + 1] (device), or nullptr
    int32_t rows;         // varlen segment launches: rows launched (an upper bound)
    int32_t s0_bf16;      // 1: s0 holds bf16 values (same layout), else fp32
    int32_t sfin_bf16;    // 1: sfin is written as bf16 (round to nearest even), else fp32
};

// The recurrent decode step: T tokens of each of N dense sequences, H heads.
struct DecodeParams {
    const __nv_bfloat16* q;   // [N][T][H][128]
    const __nv_bfloat16* k;
    const __nv_bfloat16* v;
    const float* g;
    const __nv_bfloat16* beta;  // [N][T][H]
    const void* s0;           // [N][H][128][128] fp32 or bf16 (state_bf16), or nullptr
    void* sfin;               // same layout and type, or nullptr; may equal s0
    __nv_bfloat16* out;       // [N][T][H][128]
    int64_t T;
    int32_t N;
    int32_t H;                // heads of v, g, beta and the states
    int32_t Hq;               // heads of q; see HeadMap
    float scale;
    int32_t state_bf16;       // 1: states are bf16, else fp32
};

// Grouped heads.  H state heads (v, g, beta, states), Hq query heads, min(Hq, H) key
// heads and Ho = max(Hq, H) output heads, one of the two a multiple of the other.
// Output head ho reads q head hq, k head hk and state head hs:
//   Hq <= H (grouped value heads): hs = ho, hq = hk = ho / (H / Hq);
//   Hq >  H (grouped query heads):  hq = ho, hs = hk = ho / (Hq / H); the Hq / H output
//           heads of a state head run the same chain, and the first writes its state.
struct HeadMap {
    int hq, hk, hs;
    bool state_owner;
};
__host__ __device__ inline HeadMap head_map(int ho, int H, int Hq) {
    HeadMap m;
    if (Hq <= H) {
        m.hs = ho;
        m.hq = m.hk = ho / (H / Hq);
        m.state_owner = true;
    } else {
        const int G = Hq / H;
        m.hq = ho;
        m.hs = m.hk = ho / G;
        m.state_owner = (ho % G) == 0;
    }
    return m;
}

// Launch flags of the fused kernel.
constexpr int32_t kFlagNoOutput = 1;       // no output rows (summary runs)
constexpr int32_t kFlagZeroV = 2;          // treat v as zero (transition runs: U = 0)
constexpr int32_t kFlagIdentityS0 = 4;     // initial state = identity
constexpr int32_t kFlagFinalLastSeg = 8;   // write final state only for the last segment, at its sequence
constexpr int32_t kFlagSkipLastSeg = 16;   // varlen summaries: the last segment of a sequence is not run

// Token range [bos, eos) of sequence n; false (and the status word set) when
// cu_seqlens is malformed for this sequence.
// Token range of CTA row n, with its sequence, segment index and the sequence's segment
// count (1 and 0 outside segment launches).  False: nothing to run for this row.
__device__ __forceinline__ bool seq_range(const FwdParams& p, int n, int64_t& bos, int64_t& eos,
                                          int& seq, int& sg, int& nsg) {
    seq = n;
    sg = 0;
    nsg = 1;
    if (p.seg_len > 0 && p.cu == nullptr) {
        seq = n / p.nseg_used;
        sg = n % p.nseg_used;
        nsg = p.nseg_total;
        const int64_t base = (int64_t)seq * p.dense_len;
        const int64_t a = (int64_t)sg * p.seg_len;
        bos = base + a;
        eos = base + (a + p.seg_len < p.dense_len ? a + p.seg_len : p.dense_len);
        return true;
    }
    if (p.seg_len > 0) {
        if (n >= p.seg_start[p.N]) return false;
        int lo = 0, hi = p.N - 1;  // last sequence whose first row is <= n
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (p.seg_start[mid] <= n) lo = mid;
            else hi = mid - 1;
        }
        seq = lo;
        sg = n - p.seg_start[lo];
        nsg = p.seg_start[lo + 1] - p.seg_start[lo];
        if ((p.flags & kFlagSkipLastSeg) && sg == nsg - 1) return false;
        const int64_t end = p.cu[seq + 1];
        bos = p.cu[seq] + (int64_t)sg * p.seg_len;
        eos = bos + p.seg_len < end ? bos + p.seg_len : end;
        return true;
    }
    if (p.cu == nullptr) {
        bos = (int64_t)n * p.dense_len;
        eos = bos + p.dense_len;
        return true;
    }
    bos = p.cu[n];
    eos = p.cu[n + 1];
    if ((n == 0 && bos != 0) || bos < 0 || eos < bos || eos > p.T_total) {
        atomicCAS(p.status, kStatusOk, kStatusBadSeqlens);
        return false;
    }
    return true;
}

// TMA descriptors of the [T_total][H][128] inputs, box {128, 1, 16} (one chunk of
// one head).  Encoded on the host, passed to kernels as __grid_constant__ params.
struct TensorMaps {
    CUtensorMap q, k, v, g;
    CUtensorMap out;  // output (TMA stores of full chunks)
};

// Launchers (return the launch error, cudaSuccess on success).
// Fused K1+K2 kernel over p.N x max(p.Hq, p.H) rows (or the segment rows of a segment
// launch, which need Hq == H).
cudaError_t launch_serial(const FwdParams& p, const TensorMaps& maps, cudaStream_t stream);
// Segment merge: carry[b][0] = S0[b] (or 0), carry[b][s+1] = m[b][s] carry[b][s] + bs[b][s].
// Varlen segment table: seg_start[n] = sum over sequences before n of
// max(1, ceil(len / seg_len)); validates cu_seqlens (status word on malformed input).
cudaError_t launch_segment_table(const int32_t* cu, int32_t N, int64_t T_total, int64_t seg_len,
                                 int32_t* seg_start, int32_t* status, cudaStream_t stream);
// Dense: B sequences of nseg segments.  Varlen (seg_start != nullptr): B = N sequences,
// each with its own count from the table; summaries and carries indexed by segment row.
// The carry's columns are split over merge_block_cols(B, H, sm_count)-wide blocks.
// s0: fp32, or bf16 when s0_bf16 (the caller's initial states); carries stay fp32.
cudaError_t launch_merge(const float* m_seg, const float* b_seg, const void* s0, int s0_bf16, float* carries,
                         int32_t B, int32_t nseg, int32_t H, int sm_count, cudaStream_t stream,
                         const int32_t* seg_start = nullptr);
int merge_block_cols(int32_t B, int32_t H, int sm_count);
cudaError_t merge_init();  // shared-memory limits of the merge kernels, once per device
// Decode: one CTA per (sequence, head).
cudaError_t launch_decode(const DecodeParams& p, cudaStream_t stream);
size_t serial_smem_bytes();
int serial_block_threads();
const void* serial_kernel_symbol();   // equal head counts
const void* grouped_kernel_symbol();  // grouped heads (same shared memory and block size)

}  // namespace kda
