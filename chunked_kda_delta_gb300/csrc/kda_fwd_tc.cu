// kda_fwd_tc.cu -- fused K1 + K2 KDA forward prefill for sm_103a: one 2-CTA thread-block
// cluster per (sequence, head); TMA-staged chunk tiles; tcgen05 MMAs with the state held
// in tensor memory (TMEM) across all chunks.
//
// The method (cuLA PR #103 "feat(kda/sm90): FlashKDA prefill port + intracard-CP
// prefill", commit notes): two stages, forward only, chunks of 16 tokens and head size
// 128; K1 builds the decayed q/k, applies beta and forms the WY inverse of each chunk,
// and K2 carries the state from chunk to chunk.  For a chunk of C <= 16
// rows with chunk-start state S (Dk x Dv = 128 x 128) and in-chunk cumulative
// log-decay gam_r = sum_{m<=r} g_m (per channel):
//   A      = strict_lower(beta_r (k_r . k_s exp(gam_r - gam_s)))      16x16
//   Tb     = (I + A)^{-1} diag(beta)                                   WY inverse
//   W      = Tb (K o exp(gam)),   U = Tb V                             16x128
//   Mq     = lower(q_r . k_s exp(gam_r - gam_s))                       16x16
//   delta  = U - W S
//   O      = scale (Qtil S + Mq delta),  Qtil = Q o exp(gam)
//   S     <- Diag(exp gam_C) S + Kbar^T delta,  Kbar_r = k_r o exp(gam_C - gam_r)
// exp(gam_r - gam_s) is factored through the chunk's row 7 as
// exp(gam_r - gam_ref) exp(gam_ref - gam_s), and K o exp(gam), Q o exp(gam) are formed as
// (K o exp(gam - gam_ref)) exp(gam_ref).  Each factor is at most e^kFastLimit while a
// channel's cumulative log-decay falls by at most kFastLimit over the chunk.  A chunk with
// channels beyond that (strong decay) takes strong_decay_chunk() as well: those channels
// leave the factored Grams, their terms k_r k_s exp(gam_r - gam_s) (q_r for Mq) are
// formed pair by pair with the exponent taken directly, and their K o exp(gam),
// Q o exp(gam) and Kbar are formed directly, so no factor exceeds 1 for g <= 0.
//
// Mapping (transposed so the 128-wide value dim is the MMA's M):
//   TMEM holds S^T (lane j = value column, column i = key row) in fp32.
//   One-chunk lookahead: with D_c = Diag(exp gam_C(c-1)) S_{c-1},
//     W_c S_c = W_c D_c + P_{c-1} delta_{c-1},  P_{c-1} = W_c Kbar_{c-1}^T (Qtil, R alike),
//   so MMA1 of chunk c (A = bf16 D_c^T in TMEM, B = [W ; Qtil]) needs only D_c.  Its
//   accumulator also collects delta_{c-1}^T [P ; R]^T, hence
//     delta_c^T = U_c^T - (sum of the W partials),  O_c = scale (sum of the Qtil partials + Mq delta).
//   MMA2: S^T += delta^T . Kbar, after the chain scaled S^T by exp(gam_C) in place.
//
// Work split (416 threads per CTA, 13 warps):
//   CTA rank 0 ("K1 CTA"): warp 0 is the TMA producer (q/k/v/g tiles into a ring with
//     one stage per K1 group; beta with plain loads, two chunks ahead); warps 1-12 are
//     three K1 groups of 4 warps taking every third chunk (cumulative decay, decayed
//     operands, in-chunk Grams and the WY solve, W and U; the 16x16 products use mma.sync
//     because tcgen05's smallest M is 64).  A group writes its chunk's operands (21.8 KB)
//     into one of four local stages and ships them to the K2 CTA with one
//     cp.async.bulk shared::cta -> shared::cluster copy that completes the K2 CTA's
//     barrier.
//   CTA rank 1 ("K2 CTA"): warps 1-8 run the state chain (decay and bf16 copy of the
//     state, delta, output rows) and only arrive on two named barriers; warp 11 issues
//     the state update and the Mq term, warps 10 and 9 MMA1 of the next chunk (the
//     tensor pipe runs one thread's MMAs in order but overlaps different threads'), warp
//     9 also issues the output tiles' TMA stores; warp 12 computes [P ; R] ahead of the
//     chain; warp 0 owns TMEM, relays copy landings back to the K1 groups and publishes
//     how many chunks have landed.
// Splitting a chain over two SMs doubles the shared-memory bandwidth and issue slots
// each chunk gets; one SM alone was bound by its shared-memory pipe.
// Every wait is bounded: on exhaustion the kernel records KDA_ERR_DEVICE_TIMEOUT in the
// status word, drains its in-flight copies and MMAs, meets its peer at the final
// cluster barrier and exits.
#include <cuda.h>

#include "kda_internal.cuh"
#include "kda_ptx.cuh"

namespace kda {
namespace {

using namespace ptx;

constexpr int kK1Groups = 3;                    // K1 groups, chunk c -> group c % 3
constexpr int kThreads = 32 * (1 + 4 * kK1Groups);  // 416
constexpr int kRef = 7;
constexpr float kFastLimit = 80.f;  // largest log-decay fall over a chunk for the factored path
constexpr uint32_t kTmemCols = 512;
// Bound of the waits that drain in-flight copies and MMAs before exit; independent of
// the caller's wait limit so that an early exit never leaves asynchronous work behind.
constexpr int64_t kDrainLimit = 1ll << 22;  // rounds of at most ~1 us each
constexpr float kLog2e = 1.4426950408889634f;

// TMEM column map (K2 CTA)
constexpr uint32_t kColS = 0;     // S^T fp32, 128 columns
constexpr uint32_t kColSA = 128;  // S^T bf16 pairs, 64 columns (MMA1 A operand)
// MMA1 accumulators: 2 buffers x 2 K-half partials x 32 columns; in each partial,
// columns 0-15 hold D^T W^T and 16-31 hold D^T Qtil^T; partial 0 also collects the
// lookahead terms delta^T [P ; R]^T of the previous chunk and delta^T Mq^T.
constexpr uint32_t kColD1 = 192;
constexpr uint32_t kD1Buf = 64;   // columns per MMA1 buffer
constexpr uint32_t kColDA = 320;  // 2 buffers x 8 columns: delta^T bf16 pairs (A operand)

// Input stage (K1 CTA): q, k, v bf16 [16][128]; g fp32 [16][128]; beta fp32 [16].
constexpr int kInQ = 0, kInK = 4096, kInV = 8192, kInG = 12288, kInBeta = 20480;
constexpr int kInBytes = 20608;
// One input stage per K1 group (chunk c -> stage c % 3 = group c % 3): successive phases
// of a stage's barriers then belong to one group, in order, so a group never waits on a
// phase two ahead of the last one it saw complete (a parity wait cannot tell those apart).
constexpr int kInStages = kK1Groups;
constexpr uint32_t kTxBytes = 20480;  // q, k, v, g tiles
// Chunk operand stage (K1 -> K2): B1 = [W ; Qtil] (N=32, K=128), B2 = Kbar (N=128,
// K=16), B3 = Mq (N=16, K=16), all bf16 in the no-swizzle K-major layout; U fp32 rows
// padded to 132 floats so the fragment-layout float2 stores hit 32 distinct banks;
// exp(gam_C) fp32 [128].
constexpr int kURow = 132;
constexpr int kB1 = 0, kB2 = 8192, kB3 = 12288, kU = 12800, kGC = kU + 16 * kURow * 4,
              kOutBytes = kGC + 512;
// Receive ring: two stages per K1 group (chunk c -> stage c % 6, group c % 3), so a stage
// is only refilled by the group that filled it last and its release barrier is never
// more than one phase behind that group.
constexpr int kRecvStages = 2 * kK1Groups;
constexpr uint32_t kLbo = 128, kSboB1 = 2048, kSboB2 = 256, kSboB3 = 256;
// K1 group scratch: padded bf16 staging rows (136 elements), exp(gam_ref), A, Tb, beta.
constexpr int kStRow = 272, kStArr = 16 * kStRow;
enum { ST_KQ = 0, ST_QQ, ST_KK, ST_VV, ST_NUM };
// Strong-decay chunks also use: a flag word and the 128-bit channel mask, and the exact
// Gram terms (A^T, then Mq^T, fp32 [16][16] each).
constexpr int kGEref = ST_NUM * kStArr, kGA = kGEref + 512, kGTb = kGA + 1024,
              kGBeta = kGTb + 768, kGSlow = kGBeta + 64, kGCorr = kGSlow + 32,
              kGrpBytes = kGCorr + 2048;
// Shared memory map.  K1 CTA: input ring, the group scratches, the local operand stages.
// K2 CTA: receive ring at offset 0.  Barriers sit at the same offset in both.
constexpr int kSmIn = 0;
constexpr int kSmGrp = kSmIn + kInStages * kInBytes;
constexpr int kSmOutLocal = kSmGrp + kK1Groups * kGrpBytes;
// Local operand stages (K1 CTA), chunk c -> stage c % kOutStages, shared by the groups
// round-robin: a group writes chunk c's operands once the copy of chunk c - kOutStages
// has landed.  The relay reports landings in chunk order, so when a group waits for that
// copy it has already seen chunk c - kOutStages - 1 land (its own previous chunk's stage
// wait covered it): the stage barrier is never waited on two phases ahead.
constexpr int kOutStages = kK1Groups + 1;
constexpr int kSmRecv = 0;
constexpr int kSmOTile = kSmRecv + kRecvStages * kOutBytes;  // K2 CTA: output tiles bf16 [16][128]
constexpr int kOTileBytes = kChunk * kD * 2;
constexpr int kOTiles = 4;  // output tiles: a tile is rewritten 4 chunks after its store
// K2 CTA: ring of [P ; R] lookahead operands (bf16, N = 32 x K = 16, K-major):
// P_c = W_{c+1} Kbar_c^T, R_c = Qtil_{c+1} Kbar_c^T.
constexpr int kSmPR = kSmOTile + kOTiles * kOTileBytes;
constexpr int kPRBytes = 1024;
constexpr int kPRSlots = 3;
constexpr int kSmBar = kSmOutLocal + kOutStages * kOutBytes;
constexpr int kNumBars = 24;
constexpr int kSmTmemSlot = kSmBar + kNumBars * 8;
constexpr int kSmFail = kSmTmemSlot + 8;            // int32 per K1 group: failure flags
constexpr int kSmK2Fail = kSmFail + 4 * kK1Groups;  // int32: K2 CTA failure flag
constexpr int kSmLanded = kSmK2Fail + 4;            // int32: K2 CTA, chunks landed so far
constexpr int kSmPrReady = kSmLanded + 4;           // int32: K2 CTA, [P ; R] operands written
constexpr int kSmPrUsed = kSmPrReady + 4;           // int32: K2 CTA, [P ; R] operands consumed
constexpr int kSmemBytes = kSmPrUsed + 4;
static_assert(kSmPR + kPRSlots * kPRBytes <= kSmBar, "K2 buffers overlap the barriers");
static_assert(kSmOTile % 128 == 0, "TMA store source must be 128-byte aligned");
enum {  // K1 CTA barriers
    BAR_IN_FULL = 0, BAR_IN_EMPTY = 4, BAR_OUT_FREE = 8,
    BAR_COPIED = BAR_OUT_FREE + kRecvStages  // per local operand stage: its last bulk copy has landed
};
static_assert(kInStages <= BAR_IN_EMPTY - BAR_IN_FULL, "input barriers overlap");
static_assert(BAR_COPIED + kOutStages <= kNumBars, "too many barriers");
enum {  // K2 CTA barriers
    BAR_K1_FULL = 0,                       // kRecvStages: chunk operands landed
    BAR_D1 = BAR_K1_FULL + kRecvStages,    // MMA1 group of a chunk complete (2 commits)
    BAR_SDONE,                             // state update and Mq delta complete (1 commit)
    BAR_DRAIN,                             // every MMA complete before exit (3 issuers)
    BAR_NEVER,                             // never signalled (timeout-path test)
    BAR_PR_FULL,                           // kPRSlots: [P ; R] operand written
    BAR_PR_FREE = BAR_PR_FULL + kPRSlots,  // kPRSlots: [P ; R] operand consumed
    BAR_K2_END = BAR_PR_FREE + kPRSlots
};
static_assert(BAR_K2_END <= kNumBars, "too many barriers");
// K2 CTA named barriers (the K1 CTA uses 1 .. kK1Groups in its own CTA): the state
// chain (8 warps) arrives, the MMA issuers wait.
constexpr uint32_t kNamedIssue = 1;  // delta_c and D_{c+1} written: state update, Mq
constexpr uint32_t kNamedEmit = 2;   // output of chunk c-1 read, bf16 D_{c+1} written: MMA1(c+1)
constexpr uint32_t kChainThreads = 256, kIssueCount = kChainThreads + 32, kEmitCount = kChainThreads + 64;
// K2 CTA roles outside the chain (warps 1-8).  A warp runs on SM sub-partition
// warp % 4: the two MMA1 issuers (10, 9) sit on different ones, so they issue in parallel,
// and the busy [P ; R] warp shares sub-partition 0 with the nearly idle relay.
constexpr int kRelayWarp = 0;      // copy relay (and the TMEM allocation)
constexpr int kPRWarp = 12;        // [P ; R] operands
constexpr int kUpdateWarp = 11;    // state update and output term
constexpr int kMma1WarpA = 10;     // MMA1 keys 0-63 and the lookahead term
constexpr int kMma1WarpB = 9;      // MMA1 keys 64-127 and the output tiles' TMA stores

__device__ __forceinline__ uint32_t b1_off(int n, int k) {
    return (n >> 3) * kSboB1 + (k >> 3) * kLbo + (n & 7) * 16 + (k & 7) * 2;
}
__device__ __forceinline__ uint32_t b3_off(int n, int k) {
    return (n >> 3) * kSboB3 + (k >> 3) * kLbo + (n & 7) * 16 + (k & 7) * 2;
}

__device__ __forceinline__ void record(int32_t* status, int32_t code) {
    atomicCAS(status, kStatusOk, code);
}

// A chunk with strong-decay channels (a channel whose cumulative log-decay falls by more
// than kFastLimit over the chunk), run by the 128 threads of its K1 group after phase 1
// and before phase 2; `t` = thread in the group, (pc, hr) its channel pair and row half
// as in phase 1.  Phase 1 has already written the factored operands of every channel;
// this pass
//   - turns g in the input stage into the cumulative log-decay gam (rows past C add 0),
//   - for each strong-decay channel c: stages K o exp(gam) and Q o exp(gam) (eref 1),
//     zero in the Gram's right operand (so the factored Grams leave c out), and writes
//     Kbar = K o exp(gam_C - gam) into B2; and records c in the channel mask,
//   - writes the exact Gram terms of the masked channels into corr:
//       corr[s * 16 + r]       = beta_r sum_c k_r[c] k_s[c] exp(gam_r[c] - gam_s[c]), s < r
//       corr[256 + s * 16 + r] = sum_c q_r[c] k_s[c] exp(gam_r[c] - gam_s[c]),      s <= r
//     (every other entry 0), which phase 2 adds to the factored Grams.
// No factor formed here exceeds 1 for g <= 0.  Ends with the group's barrier passed.
__device__ __noinline__ void strong_decay_chunk(unsigned char* in, unsigned char* grp, unsigned char* ob, int C,
                                                int t, uint32_t nbar) {
    const int pc = t & 63, hr = t >> 6;
    unsigned char* st = grp;
    float* eref = reinterpret_cast<float*>(grp + kGEref);
    unsigned char* b2 = ob + kB2;
    uint32_t* mask = reinterpret_cast<uint32_t*>(grp + kGSlow) + 4;
    float* corr = reinterpret_cast<float*>(grp + kGCorr);
    const float* beta = reinterpret_cast<const float*>(grp + kGBeta);
    float* gam = reinterpret_cast<float*>(in + kInG);
    const __nv_bfloat16* q = reinterpret_cast<const __nv_bfloat16*>(in + kInQ);
    const __nv_bfloat16* k = reinterpret_cast<const __nv_bfloat16*>(in + kInK);
    if (t < 4) mask[t] = 0u;
    reinterpret_cast<float4*>(corr)[t] = make_float4(0.f, 0.f, 0.f, 0.f);
    named_bar_sync(nbar, 128);  // every thread has read g in phase 1
    if (hr == 0) {
        float2 a = make_float2(0.f, 0.f);
        float2* g2 = reinterpret_cast<float2*>(gam);
        for (int r = 0; r < kChunk; ++r) {
            a = add2(a, r < C ? g2[r * 64 + pc] : make_float2(0.f, 0.f));
            g2[r * 64 + pc] = a;
        }
    }
    named_bar_sync(nbar, 128);
    for (int e = 0; e < 2; ++e) {
        const int c = 2 * pc + e;
        const float gc = gam[(kChunk - 1) * kD + c];
        if (gam[c] - gc <= kFastLimit) continue;
        if (hr == 0) {
            atomicOr(mask + (c >> 5), 1u << (c & 31));
            eref[c] = 1.f;
        }
        for (int rr = 0; rr < 8; ++rr) {
            const int r = 8 * hr + rr;
            const bool valid = r < C;
            const float kr = valid ? __bfloat162float(k[r * kD + c]) : 0.f;
            const float qr = valid ? __bfloat162float(q[r * kD + c]) : 0.f;
            const float gr = gam[r * kD + c];
            const float eg = ex2(gr * kLog2e), egc = ex2((gc - gr) * kLog2e);
            __nv_bfloat16* row = reinterpret_cast<__nv_bfloat16*>(st + r * kStRow) + c;
            row[ST_KQ * kStArr / 2] = __float2bfloat16_rn(kr * eg);
            row[ST_QQ * kStArr / 2] = __float2bfloat16_rn(qr * eg);
            row[ST_KK * kStArr / 2] = __float2bfloat16_rn(0.f);
            *reinterpret_cast<__nv_bfloat16*>(b2 + (c >> 3) * kSboB2 + hr * kLbo + (c & 7) * 16 + rr * 2) =
                __float2bfloat16_rn(kr * egc);
        }
    }
    named_bar_sync(nbar, 128);
    // Exact terms: pairs 0 .. 119 of A (s < r), 120 .. 255 of Mq (s <= r), rows in order.
    for (int idx = t; idx < 256; idx += 128) {
        const bool is_q = idx >= 120;
        const int pi = is_q ? idx - 120 : idx;
        int r = is_q ? 0 : 1, base = 0;
        while (base + (is_q ? r + 1 : r) <= pi) {
            base += is_q ? r + 1 : r;
            ++r;
        }
        const int sc = pi - base;
        if (r >= C || sc >= C) continue;
        const __nv_bfloat16* a = is_q ? q : k;
        float acc = 0.f;
        for (int w = 0; w < 4; ++w) {
            uint32_t m = mask[w];
            while (m != 0u) {
                const int c = 32 * w + __ffs(m) - 1;
                m &= m - 1u;
                const float f = ex2((gam[r * kD + c] - gam[sc * kD + c]) * kLog2e);
                acc = fmaf(__bfloat162float(a[r * kD + c]) * __bfloat162float(k[sc * kD + c]), f, acc);
            }
        }
        if (is_q) corr[256 + sc * 16 + r] = acc;
        else corr[sc * 16 + r] = beta[r] * acc;
    }
    fence_proxy_async_smem();  // B2 is shipped by a bulk copy
    named_bar_sync(nbar, 128);
}

// C[r][s] = sum_c A[r][c] B[s][c] for 16x16 tiles over 128 channels; A and B are
// bf16 [16][136] staging arrays.  Four independent accumulator chains.
__device__ __forceinline__ void gram16(uint32_t abase, uint32_t bbase, int lane, float (&c)[2][4]) {
    float acc[2][2][4];
#pragma unroll
    for (int i = 0; i < 2; ++i)
#pragma unroll
        for (int j = 0; j < 2; ++j)
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[i][j][e] = 0.f;
#pragma unroll
    for (int k0 = 0; k0 < 128; k0 += 16) {
        const int kp = (k0 >> 4) & 1;
        uint32_t a0, a1, a2, a3, b0, b1, b2, b3;
        ldsm_x4(abase + (lane & 15) * kStRow + (k0 + 8 * (lane >> 4)) * 2, a0, a1, a2, a3);
        ldsm_x4(bbase + ((lane & 7) + 8 * (lane >> 4)) * kStRow + (k0 + 8 * ((lane >> 3) & 1)) * 2,
                b0, b1, b2, b3);
        mma_16816(acc[kp][0], a0, a1, a2, a3, b0, b1);
        mma_16816(acc[kp][1], a0, a1, a2, a3, b2, b3);
    }
#pragma unroll
    for (int j = 0; j < 2; ++j)
#pragma unroll
        for (int e = 0; e < 4; ++e) c[j][e] = acc[0][j][e] + acc[1][j][e];
}

// kGrouped: unequal head counts (HeadMap); the equal-count instance keeps the plain
// head indexing, which leaves the state chain two registers it needs.
template <bool kGrouped>
__global__ void __launch_bounds__(kThreads, 1)
kda_fwd_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_g,
                  const __grid_constant__ CUtensorMap tm_out, const FwdParams p) {
    extern __shared__ __align__(1024) unsigned char smem[];
    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const uint32_t rank = cluster_ctarank();   // 0: K1 CTA, 1: K2 CTA
    // (row, output head) of this cluster; the roles below look up their other heads
    const int Ho0 = kGrouped ? (p.Hq > p.H ? p.Hq : p.H) : p.H;
    const int n = (int)((blockIdx.x >> 1) / Ho0);
    const int h = kGrouped ? head_map((int)((blockIdx.x >> 1) % Ho0), p.H, p.Hq).hs
                           : (int)((blockIdx.x >> 1) % Ho0);  // state head
    int64_t bos, eos;
    int seq_id, seg_id, seg_count;
    if (!seq_range(p, n, bos, eos, seq_id, seg_id, seg_count)) return;  // both CTAs return
    const int64_t H = p.H;
    const int nchunks = (int)((eos - bos + kChunk - 1) / kChunk);
    const int64_t lim = p.wait_limit;
    const uint32_t sbase = smem_u32(smem);
    const uint32_t bars = sbase + kSmBar;
    auto bar = [&](int i) { return bars + 8u * (uint32_t)i; };
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kSmTmemSlot);
    volatile int32_t* fail_flag = reinterpret_cast<volatile int32_t*>(smem + kSmFail);

    if (tid == 0) {
        if (rank == 0) {
            for (int s = 0; s < kInStages; ++s) {
                mbar_init(bar(BAR_IN_FULL + s), 1);
                mbar_init(bar(BAR_IN_EMPTY + s), 1);
            }
            for (int s = 0; s < kRecvStages; ++s) mbar_init(bar(BAR_OUT_FREE + s), 1);
            for (int os = 0; os < kOutStages; ++os) mbar_init(bar(BAR_COPIED + os), 1);
            for (int gi = 0; gi < kK1Groups; ++gi) fail_flag[gi] = 0;
        } else {
            for (int s = 0; s < kRecvStages; ++s) mbar_init(bar(BAR_K1_FULL + s), 1);
            mbar_init(bar(BAR_D1), 2);
            mbar_init(bar(BAR_SDONE), 1);
            mbar_init(bar(BAR_DRAIN), 3);
            *reinterpret_cast<volatile int32_t*>(smem + kSmK2Fail) = 0;
            *reinterpret_cast<volatile int32_t*>(smem + kSmLanded) = 0;
            *reinterpret_cast<volatile int32_t*>(smem + kSmPrReady) = 0;
            *reinterpret_cast<volatile int32_t*>(smem + kSmPrUsed) = 0;
            mbar_init(bar(BAR_NEVER), 1);
            for (int s = 0; s < kPRSlots; ++s) {
                mbar_init(bar(BAR_PR_FULL + s), 1);
                mbar_init(bar(BAR_PR_FREE + s), 1);
            }
        }
        fence_mbar_init();
    }
    if (rank == 1 && warp == 0) {
        tmem_alloc(smem_u32(tmem_slot), kTmemCols);
        tmem_relinquish();
    }
    if (rank == 0 && warp == 0 && lane == 0 && nchunks > 0) {
        prefetch_tmap(&tm_q);
        prefetch_tmap(&tm_k);
        prefetch_tmap(&tm_v);
        prefetch_tmap(&tm_g);
    }
    tc_fence_before();
    cluster_sync();  // barriers of both CTAs initialised before any remote access
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    const uint32_t tmem = tmem_base;

    if (rank == 0 && warp == 0) {
        // ------------------------------------------------------------ TMA producer
        // beta is read with plain loads two chunks ahead (its [T][H] rows are 2 bytes
        // wide, below the 16-byte TMA granule) and stored next to the TMA tiles.  The raw
        // bf16 bits of chunks c and c + 1 sit in two registers (the loop is unrolled by
        // two) until their store: no instruction reads a load result before the load has
        // had two chunks to complete.  Widening at the load, or rotating one register
        // into another, would make this warp wait a full global-load latency on every
        // chunk, and its TMA issue rate would then bound every stage of the pipeline.
        auto load_beta = [&](int cc, uint32_t& bits) {
            bits = 0u;
            const int64_t t = bos + (int64_t)cc * kChunk + lane;
            if (lane < kChunk && cc < nchunks && t < eos)
                bits = *reinterpret_cast<const unsigned short*>(p.beta + (t * H + h));
        };
        uint32_t b_even, b_odd;
        load_beta(0, b_even);
        load_beta(1, b_odd);
        int hq = h, hk = h;  // q and k heads of this cluster, once
        if (kGrouped) {
            const HeadMap hm = head_map((int)((blockIdx.x >> 1) % (p.Hq > p.H ? p.Hq : p.H)), p.H, p.Hq);
            hq = hm.hq;
            hk = hm.hk;
        }
        int issued = 0;
        // Chunk c: wait for its input stage, store its beta (`bits`), load the beta of
        // chunk c + 2 into `bits`, issue the four tiles.  False after a timeout.
        auto produce = [&](int c, uint32_t& bits) -> bool {
            const int s = c % kInStages;
            const bool ok = c < kInStages ||
                            mbar_wait(bar(BAR_IN_EMPTY + s), ((c / kInStages) - 1) & 1, lim);
            if (__any_sync(0xffffffffu, !ok)) {
                if (lane == 0) record(p.status, kStatusTimeout);
                return false;
            }
            const uint32_t dst = sbase + kSmIn + s * kInBytes;
            if (lane < kChunk)
                reinterpret_cast<float*>(smem + kSmIn + s * kInBytes + kInBeta)[lane] = __uint_as_float(bits << 16);
            load_beta(c + 2, bits);
            __syncwarp();
            if (lane == 0) {
                const int32_t t0 = (int32_t)(bos + (int64_t)c * kChunk);
                mbar_arrive_expect_tx(bar(BAR_IN_FULL + s), kTxBytes);
                tma_load_3d(dst + kInQ, &tm_q, bar(BAR_IN_FULL + s), 0, hq, t0);
                tma_load_3d(dst + kInK, &tm_k, bar(BAR_IN_FULL + s), 0, hk, t0);
                tma_load_3d(dst + kInV, &tm_v, bar(BAR_IN_FULL + s), 0, h, t0);
                tma_load_3d(dst + kInG, &tm_g, bar(BAR_IN_FULL + s), 0, h, t0);
            }
            issued = c + 1;
            return true;
        };
        for (int c = 0; c < nchunks; c += 2) {
            if (!produce(c, b_even)) break;
            if (c + 1 < nchunks && !produce(c + 1, b_odd)) break;
        }
        // Drain: every issued load must have landed before the CTA exits.
        if (lane == 0)
            for (int c = (issued >= kInStages ? issued - kInStages : 0); c < issued; ++c)
                if (!mbar_wait(bar(BAR_IN_FULL + (c % kInStages)), (c / kInStages) & 1, kDrainLimit))
                    record(p.status, kStatusTimeout);
    } else if (rank == 0) {
        // ------------------------------------------------------------ K1 groups (kK1Groups x 128 threads)
        const int gi = (warp - 1) >> 2;   // group: chunks c with c % kK1Groups == gi
        const uint32_t nbar = 1 + gi;     // named barrier of the group
        const int kt = tid - 32 - 128 * gi;
        const int kw = kt >> 5;           // warp within the group
        // Phase-2 role of this warp, rotated by group: a CTA's warp w runs on SM
        // sub-partition w % 4, so rotating puts the three groups' solve warps (role 0) on
        // sub-partitions 1, 2 and 3 (the producer has 0) and their Mq warps next to them.
        const int kr = (kw - gi) & 3;
        // The thread that waits on the group's barriers (input tiles, previous copy) is
        // lane 0 of the group's warp (gi + 1) % 3: sub-partitions 2, 3 and 1 for groups 0,
        // 1 and 2, and never the solve warp (gi) nor the shipping warp (3).
        const int kt_wait = 32 * ((gi + 1) % 3);
        const int pc = kt & 63;           // channel pair: channels 2pc, 2pc+1
        const int hr = kt >> 6;           // row half: rows 8hr .. 8hr+7
        unsigned char* grp = smem + kSmGrp + gi * kGrpBytes;
        unsigned char* st = grp;
        float* eref_sm = reinterpret_cast<float*>(grp + kGEref);
        float* Asm = reinterpret_cast<float*>(grp + kGA);
        __nv_bfloat16* Tb = reinterpret_cast<__nv_bfloat16*>(grp + kGTb);
        float* bet = reinterpret_cast<float*>(grp + kGBeta);
        // Strong-decay chunks: flag word (set by any thread of the group in phase 1, read
        // after the group's barrier), channel mask and exact Gram terms.
        volatile uint32_t* slow_flag = reinterpret_cast<volatile uint32_t*>(grp + kGSlow);
        float* corr = reinterpret_cast<float*>(grp + kGCorr);
        const float2 l2e2 = make_float2(kLog2e, kLog2e), nl2e2 = make_float2(-kLog2e, -kLog2e);
        const bool zero_v = (p.flags & kFlagZeroV) != 0;
        const bool with_out = (p.flags & kFlagNoOutput) == 0;
        for (int c = gi; c < nchunks; c += kK1Groups) {
            const int s = c % kInStages;
            // (every thread of the group is past the previous chunk's phase 2)
            if (kt == 0) *slow_flag = 0u;
            // One thread waits for the input tiles; the group barrier publishes them.
            bool ok = !fail_flag[gi];
            if (kt == kt_wait) ok = ok && mbar_wait(bar(BAR_IN_FULL + s), (c / kInStages) & 1, lim);
            if (named_bar_or(nbar, 128, !ok)) {
                if (kt == kt_wait) record(p.status, kStatusTimeout);
                break;
            }
            const int64_t t0 = bos + (int64_t)c * kChunk;
            const int C = (eos - t0 < kChunk) ? (int)(eos - t0) : kChunk;
            const unsigned char* in = smem + kSmIn + s * kInBytes;
            if (kt < kChunk) bet[kt] = reinterpret_cast<const float*>(in + kInBeta)[kt];

            // Phase 1: cumulative decay (log2 units) and decayed operands for
            // channels 2pc, 2pc+1, rows 8hr .. 8hr+7.
            const float2* g2 = reinterpret_cast<const float2*>(in + kInG);
            float2 gl[kChunk];
            {
                float2 a = make_float2(0.f, 0.f);
#pragma unroll
                for (int r = 0; r < kChunk; ++r) {
                    const float2 gv = r < C ? g2[r * 64 + pc] : make_float2(0.f, 0.f);
                    a = add2(a, gv);
                    gl[r] = a;
                }
            }
            const float2 refl = mul2f(gl[kRef], l2e2);       // gam_ref * log2(e)
            const float2 nrefl = make_float2(-refl.x, -refl.y);
            const float2 lastl = mul2f(gl[kChunk - 1], l2e2);
            const float2 ecr = ex2x2(add2(lastl, nrefl));     // exp(gam_C - gam_ref)
            const float2 gcl = ex2x2(lastl);  // exp(gam_C), written to the operand buffer below
            // (gam is non-increasing for g <= 0: its fall over the chunk is gam_0 - gam_15)
            if (gl[0].x - gl[kChunk - 1].x > kFastLimit || gl[0].y - gl[kChunk - 1].y > kFastLimit)
                *slow_flag = 1u;
            if (hr == 0) reinterpret_cast<float2*>(eref_sm)[pc] = ex2x2(refl);
            const uint32_t* q2 = reinterpret_cast<const uint32_t*>(in + kInQ);
            const uint32_t* k2 = reinterpret_cast<const uint32_t*>(in + kInK);
            const uint32_t* v2 = reinterpret_cast<const uint32_t*>(in + kInV);
            uint32_t kb0[4], kb1[4];  // Kbar rows 8hr.. of channels 2pc and 2pc+1, bf16 pairs
            float2 kbe = make_float2(0.f, 0.f);  // Kbar of the pair's even row
#pragma unroll
            for (int rr = 0; rr < 8; ++rr) {
                const int r = 8 * hr + rr;
                const bool valid = r < C;
                const float2 gr = hr ? gl[8 + rr] : gl[rr];
                const uint32_t qv = valid ? q2[r * 64 + pc] : 0u;
                const uint32_t kv = valid ? k2[r * 64 + pc] : 0u;
                const uint32_t vv = (valid && !zero_v) ? v2[r * 64 + pc] : 0u;
                const float2 kf = bf2_to_f2(kv), qf = bf2_to_f2(qv);
                const float2 up = ex2x2(fma2(gr, l2e2, nrefl));   // exp(gam_r - gam_ref)
                const float2 dn = ex2x2(fma2(gr, nl2e2, refl));   // exp(gam_ref - gam_r)
                const float2 kq = mul2f(kf, up), qq = mul2f(qf, up), kk = mul2f(kf, dn);
                const float2 kb = mul2f(kk, ecr);                  // Kbar
                uint32_t* row = reinterpret_cast<uint32_t*>(st + r * kStRow) + pc;
                row[ST_KQ * kStArr / 4] = pack_bf16(kq.x, kq.y);
                row[ST_QQ * kStArr / 4] = pack_bf16(qq.x, qq.y);
                row[ST_KK * kStArr / 4] = pack_bf16(kk.x, kk.y);
                row[ST_VV * kStArr / 4] = vv;
                if (rr & 1) {  // rows rr-1 (low half) and rr (high half) of each channel
                    kb0[rr >> 1] = pack_bf16(kbe.x, kb.x);
                    kb1[rr >> 1] = pack_bf16(kbe.y, kb.y);
                } else {
                    kbe = kb;
                }
            }
            // The local operand stage is written from here on: the bulk copy of chunk
            // c - kOutStages out of it must have landed (a copy into the peer CTA completes
            // only through the peer's barrier, which the K2 CTA relays back).  Waiting this
            // late gives that copy the whole of phase 1 to land.
            const int lst = c % kOutStages;
            unsigned char* ob = smem + kSmOutLocal + lst * kOutBytes;
            bool copied = true;
            if (kt == kt_wait && c >= kOutStages)
                copied = mbar_wait(bar(BAR_COPIED + lst), ((c / kOutStages) - 1) & 1, lim);
            if (named_bar_or(nbar, 128, !copied)) {
                if (kt == kt_wait) record(p.status, kStatusTimeout);
                break;
            }
            // (the flag was set before the barrier above: the same answer in every thread)
            const bool strong = *slow_flag != 0u;
            if (kt == kt_wait && !strong) mbar_arrive(bar(BAR_IN_EMPTY + s));  // input tiles consumed
            {   // Kbar rows 2pc, 2pc+1 of B2 (N = key channel, K = chunk row), exp(gam_C)
                unsigned char* b2 = ob + kB2;
                const int c0 = 2 * pc, c1 = 2 * pc + 1;
                *reinterpret_cast<uint4*>(b2 + (c0 >> 3) * kSboB2 + hr * kLbo + (c0 & 7) * 16) =
                    make_uint4(kb0[0], kb0[1], kb0[2], kb0[3]);
                *reinterpret_cast<uint4*>(b2 + (c1 >> 3) * kSboB2 + hr * kLbo + (c1 & 7) * 16) =
                    make_uint4(kb1[0], kb1[1], kb1[2], kb1[3]);
                if (hr == 0) reinterpret_cast<float2*>(ob + kGC)[pc] = gcl;
            }
            if (strong) {
                strong_decay_chunk(smem + kSmIn + s * kInBytes, grp, ob, C, kt, nbar);
                if (kt == kt_wait) mbar_arrive(bar(BAR_IN_EMPTY + s));  // input tiles consumed
            }

            // Phase 2 (by role kr): 0 Gram A and the WY solve; 1 Gram Mq; 2-3 write
            // Qtil = (Q o exp(gam - gam_ref)) exp(gam_ref) into rows 16..31 of B1.
            if (kr == 0 || (kr == 1 && with_out)) {
                float acc[2][4];
                gram16(smem_u32(st + (kr == 0 ? ST_KQ : ST_QQ) * kStArr),
                       smem_u32(st + ST_KK * kStArr), lane, acc);
                const int g = lane >> 2, t = lane & 3;
                if (kr == 0) {
#pragma unroll
                    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int r = g + 8 * (e >> 1), sc = 8 * nt + 2 * t + (e & 1);
                            Asm[sc * 16 + r] = sc < r ? bet[r] * acc[nt][e] : 0.f;  // A^T
                        }
                    __syncwarp();
                    if (*slow_flag != 0u) {
                        for (int i = lane; i < 256; i += 32) Asm[i] += corr[i];
                        __syncwarp();
                    }
                    if (lane < 16) {
                        // Column sc of T = (I + A)^{-1} by right-looking forward substitution:
                        // once x_m is final, x_r -= A[r][m] x_m for every r > m.  The updates
                        // of one step are independent, so the dependent chain is 15 FMAs.
                        const int sc = lane;
                        float x[kChunk];
#pragma unroll
                        for (int r = 0; r < kChunk; ++r) x[r] = r == sc ? 1.f : 0.f;
#pragma unroll
                        for (int m = 0; m < kChunk - 1; ++m) {
                            const float xm = x[m];
                            const float4* acol = reinterpret_cast<const float4*>(Asm + m * 16);
#pragma unroll
                            for (int r4 = (m + 1) >> 2; r4 < 4; ++r4) {
                                const float4 av = acol[r4];
                                if (4 * r4 + 0 > m) x[4 * r4 + 0] = fmaf(-av.x, xm, x[4 * r4 + 0]);
                                if (4 * r4 + 1 > m) x[4 * r4 + 1] = fmaf(-av.y, xm, x[4 * r4 + 1]);
                                if (4 * r4 + 2 > m) x[4 * r4 + 2] = fmaf(-av.z, xm, x[4 * r4 + 2]);
                                if (4 * r4 + 3 > m) x[4 * r4 + 3] = fmaf(-av.w, xm, x[4 * r4 + 3]);
                            }
                        }
                        const float bs = bet[sc];
#pragma unroll
                        for (int r = 0; r < kChunk; ++r) Tb[r * 24 + sc] = __float2bfloat16_rn(x[r] * bs);
                    }
                } else {
                    unsigned char* b3 = ob + kB3;
                    if (*slow_flag != 0u) {
#pragma unroll
                        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                            for (int e = 0; e < 4; ++e)
                                acc[nt][e] += corr[256 + (8 * nt + 2 * t + (e & 1)) * 16 + g + 8 * (e >> 1)];
                    }
#pragma unroll
                    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                        for (int hh = 0; hh < 2; ++hh) {
                            const int r = g + 8 * hh, sc = 8 * nt + 2 * t;
                            const float m0 = sc <= r ? acc[nt][2 * hh] : 0.f;
                            const float m1 = sc + 1 <= r ? acc[nt][2 * hh + 1] : 0.f;
                            *reinterpret_cast<uint32_t*>(b3 + b3_off(r, sc)) = pack_bf16(m0, m1);
                        }
                }
            } else if (kr >= 2 && with_out) {
                const int ct = 32 * (kr - 2) + lane;  // 0..63
                unsigned char* b1 = ob + kB1;
#pragma unroll
                for (int e = ct; e < 256; e += 64) {
                    const int r = e & 15, kg = e >> 4;  // 8 consecutive rows per 128-byte store
                    const uint4 src = *reinterpret_cast<const uint4*>(st + ST_QQ * kStArr + r * kStRow + kg * 16);
                    const float4 e0 = reinterpret_cast<const float4*>(eref_sm)[2 * kg];
                    const float4 e1 = reinterpret_cast<const float4*>(eref_sm)[2 * kg + 1];
                    const float2 x0 = mul2f(bf2_to_f2(src.x), make_float2(e0.x, e0.y));
                    const float2 x1 = mul2f(bf2_to_f2(src.y), make_float2(e0.z, e0.w));
                    const float2 x2 = mul2f(bf2_to_f2(src.z), make_float2(e1.x, e1.y));
                    const float2 x3 = mul2f(bf2_to_f2(src.w), make_float2(e1.z, e1.w));
                    *reinterpret_cast<uint4*>(b1 + b1_off(16 + r, kg * 8)) =
                        make_uint4(pack_bf16(x0.x, x0.y), pack_bf16(x1.x, x1.y),
                                   pack_bf16(x2.x, x2.y), pack_bf16(x3.x, x3.y));
                }
            }
            named_bar_sync(nbar, 128);

            // Phase 3: W = (Tb (K o exp(gam - gam_ref))) o exp(gam_ref), U = Tb V;
            // K1 warp kw owns columns [32kw, 32kw + 32).
            {
                uint32_t a0, a1, a2, a3;
                ldsm_x4(smem_u32(Tb) + (lane & 15) * 48 + 8 * (lane >> 4) * 2, a0, a1, a2, a3);
                const int g = lane >> 2, t = lane & 3;
                unsigned char* b1 = ob + kB1;
                float* U = reinterpret_cast<float*>(ob + kU);
#pragma unroll
                for (int which = 0; which < 2; ++which) {
                    const uint32_t bb = smem_u32(st + (which == 0 ? ST_KQ : ST_VV) * kStArr);
#pragma unroll
                    for (int half = 0; half < 2; ++half) {
                        const int n0 = 32 * kw + 16 * half;
                        uint32_t b0, b1r, b2, b3;
                        ldsm_x4_t(bb + ((lane & 7) + 8 * ((lane >> 3) & 1)) * kStRow +
                                      (n0 + 8 * (lane >> 4)) * 2,
                                  b0, b1r, b2, b3);
                        float d0[4] = {0.f, 0.f, 0.f, 0.f}, d1[4] = {0.f, 0.f, 0.f, 0.f};
                        mma_16816(d0, a0, a1, a2, a3, b0, b1r);
                        mma_16816(d1, a0, a1, a2, a3, b2, b3);
#pragma unroll
                        for (int nt = 0; nt < 2; ++nt) {
                            const float* d = nt ? d1 : d0;
                            const int col = n0 + 8 * nt + 2 * t;
                            if (which == 0) {
                                const float2 er = reinterpret_cast<const float2*>(eref_sm)[col >> 1];
                                const float2 w0 = mul2f(make_float2(d[0], d[1]), er);
                                const float2 w1 = mul2f(make_float2(d[2], d[3]), er);
                                *reinterpret_cast<uint32_t*>(b1 + b1_off(g, col)) = pack_bf16(w0.x, w0.y);
                                *reinterpret_cast<uint32_t*>(b1 + b1_off(g + 8, col)) = pack_bf16(w1.x, w1.y);
                            } else {
                                *reinterpret_cast<float2*>(U + g * kURow + col) = make_float2(d[0], d[1]);
                                *reinterpret_cast<float2*>(U + (g + 8) * kURow + col) = make_float2(d[2], d[3]);
                            }
                        }
                    }
                }
            }
            fence_proxy_async_smem();
            named_bar_sync(nbar, 128);
            // A thread of the group's last warp (never its solve warp: that is warp gi < 3)
            // ships the chunk while the waiting thread already waits for the next chunk's
            // input tiles.
            if (kt == 96) {
                // Ship the chunk's operands into the K2 CTA's receive stage.
                const int os = c % kRecvStages;
                bool free_ok = c < kRecvStages ||
                               mbar_wait_cluster(bar(BAR_OUT_FREE + os), ((c / kRecvStages) - 1) & 1, lim);
                if (free_ok) {
                    const uint32_t rbar = mapa(bar(BAR_K1_FULL + os), 1);
                    mbar_arrive_expect_tx_remote_relaxed(rbar, (uint32_t)kOutBytes);
                    bulk_copy_to_peer(mapa(sbase + kSmRecv + os * kOutBytes, 1), smem_u32(ob),
                                      (uint32_t)kOutBytes, rbar);
                    bulk_commit();
                } else {
                    fail_flag[gi] = 1;
                }
            }
        }
        // Copies still in flight at exit land before the K2 CTA reaches the final
        // cluster barrier (it waits for every chunk), so this CTA's memory stays valid.
    } else {
        // ------------------------------------------------------------ K2 CTA
        // Chunk c, with D_c = Diag(exp gam_C(c-1)) S_{c-1} (D_0 = S_0):
        //   W_c S_c = W_c D_c + P_{c-1} delta_{c-1},  P_{c-1} = W_c Kbar_{c-1}^T (likewise Qtil, R)
        // so the products of chunk c with the state (MMA1) run on D_c, which exists before
        // delta_{c-1} does.  Roles (all hand-offs are mbarriers or arrive/wait named barriers,
        // so no warp waits for another's unrelated work):
        //   warps 1-8   state chain: D_{c+1} = decay of S_c (fp32, and its bf16 copy),
        //               delta_c, then the output of chunk c-1;
        //   warp 11     S += Kbar_c^T delta_c and the Mq delta_c output term (after delta_c);
        //   warps 10, 9 MMA1(c+1) over the two K halves, plus the lookahead term
        //               delta_c [P_c ; R_c]^T (after the output of chunk c-1 was read);
        //               warp 9 also issues the output tiles' TMA stores;
        //   warp 12     [P_c ; R_c] with mma.sync, ahead of the chain;
        //   warp 0      tells each K1 group when its bulk copy has landed.
        volatile int32_t* k2fail = reinterpret_cast<volatile int32_t*>(smem + kSmK2Fail);
        const bool with_out = (p.flags & kFlagNoOutput) == 0;
        // Output heads and this cluster's output head, recomputed where used so that they
        // hold no registers across the chunk loop.
        auto out_heads = [&]() { return kGrouped ? (p.Hq > p.H ? p.Hq : p.H) : p.H; };
        auto out_head = [&]() { return kGrouped ? (int)((blockIdx.x >> 1) % out_heads()) : h; };
        const uint32_t idesc32 = idesc_bf16(128, 32), idesc128 = idesc_bf16(128, 128),
                       idesc16 = idesc_bf16(128, 16);
        const uint32_t idesc1 = with_out ? idesc32 : idesc16;  // MMA1 N: W and Qtil, or W only
        auto k1_full = [&](int c) {
            return mbar_wait(bar(BAR_K1_FULL + c % kRecvStages), (c / kRecvStages) & 1, lim);
        };
        auto stage = [&](int c) { return sbase + kSmRecv + (uint32_t)(c % kRecvStages) * kOutBytes; };
        // Progress counters published with release stores (relay: chunks landed; PR warp:
        // lookahead operands written); a reader that sees enough progress skips the barrier
        // wait, and otherwise falls back to it.
        int32_t* landed = reinterpret_cast<int32_t*>(smem + kSmLanded);
        int32_t* pr_ready = reinterpret_cast<int32_t*>(smem + kSmPrReady);
        int32_t* pr_used = reinterpret_cast<int32_t*>(smem + kSmPrUsed);
        auto landed_or_wait = [&](int c) { return ld_acquire_cta(landed) > c || k1_full(c); };
        if ((p.debug_flags & 1) && !mbar_wait(bar(BAR_NEVER), 0, lim)) *k2fail = 1;  // never signalled

        if (warp == kRelayWarp) {
            // ---- copy relay
            if (lane == 0) {
                for (int c = 0; c < nchunks; ++c) {
                    if (!k1_full(c)) {
                        record(p.status, kStatusTimeout);
                        *k2fail = 1;
                        break;
                    }
                    st_release_cta(landed, c + 1);
                    mbar_arrive_remote_relaxed(mapa(bar(BAR_COPIED + c % kOutStages), 0));
                }
            }
            __syncwarp();
        } else if (warp == kPRWarp) {
            // ---- [P_m ; R_m] = [W_{m+1} ; Qtil_{m+1}] Kbar_m^T (16x16 each, K = 128)
            for (int m = 0; m + 1 < nchunks; ++m) {
                const int slot = m % kPRSlots;
                bool w = !*k2fail;
                // Satisfied barrier waits cost this warp ~200 cycles each, and it works on
                // every chunk: the progress counters answer first (operands m - 3 read by
                // MMA1; chunks m and m + 1 landed), the barriers only when they lag.
                if (w && m >= kPRSlots)
                    w = ld_acquire_cta(pr_used) >= m - 2 ||
                        mbar_wait(bar(BAR_PR_FREE + slot), ((m / kPRSlots) - 1) & 1, lim);
                w = w && (ld_acquire_cta(landed) > m + 1 || (k1_full(m) && k1_full(m + 1)));
                if (__any_sync(0xffffffffu, !w)) {
                    if (lane == 0) record(p.status, kStatusTimeout);
                    break;
                }
            const uint32_t b1 = sbase + kSmRecv + ((m + 1) % kRecvStages) * kOutBytes + kB1;
            const uint32_t b2 = sbase + kSmRecv + (m % kRecvStages) * kOutBytes + kB2;
            float acc[2][2][2][4];  // [P or R][8-column tile][k parity][fragment]
#pragma unroll
            for (int a0 = 0; a0 < 2; ++a0)
#pragma unroll
                for (int a1 = 0; a1 < 2; ++a1)
#pragma unroll
                    for (int a2 = 0; a2 < 2; ++a2)
#pragma unroll
                        for (int e = 0; e < 4; ++e) acc[a0][a1][a2][e] = 0.f;
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
                const int i0 = 16 * kk;
                // B fragments of both 8-column tiles: Kbar rows s, channels i0 .. i0+15
                uint32_t bf[4];
                ldsm_x4_t(b2 + ((i0 + 8 * ((lane >> 3) & 1) + (lane & 7)) >> 3) * kSboB2 +
                              (lane >> 4) * kLbo + (lane & 7) * 16,
                          bf[0], bf[1], bf[2], bf[3]);
#pragma unroll
                for (int mt = 0; mt < 2; ++mt) {
                    if (mt == 1 && !with_out) continue;
                    uint32_t a0, a1, a2, a3;
                    ldsm_x4(b1 + b1_off(16 * mt + (lane & 7) + 8 * ((lane >> 3) & 1), i0 + 8 * (lane >> 4)),
                            a0, a1, a2, a3);
                    mma_16816(acc[mt][0][kk & 1], a0, a1, a2, a3, bf[0], bf[1]);
                    mma_16816(acc[mt][1][kk & 1], a0, a1, a2, a3, bf[2], bf[3]);
                }
            }
            unsigned char* prp = smem + kSmPR + slot * kPRBytes;
            const int g = lane >> 2, t = lane & 3;
#pragma unroll
            for (int mt = 0; mt < 2; ++mt)
#pragma unroll
                for (int nt = 0; nt < 2; ++nt) {
                    const float* x0 = acc[mt][nt][0];
                    const float* x1 = acc[mt][nt][1];
                    const int sc = 8 * nt + 2 * t;
                    *reinterpret_cast<uint32_t*>(prp + mt * 512 + b3_off(g, sc)) =
                        pack_bf16(x0[0] + x1[0], x0[1] + x1[1]);
                    *reinterpret_cast<uint32_t*>(prp + mt * 512 + b3_off(g + 8, sc)) =
                        pack_bf16(x0[2] + x1[2], x0[3] + x1[3]);
                }
            fence_proxy_async_smem();
            __syncwarp();
                if (lane == 0) {
                    mbar_arrive(bar(BAR_PR_FULL + slot));
                    st_release_cta(pr_ready, m + 1);
                }
            }
        } else if (warp == kUpdateWarp) {
            // ---- state update S += Kbar_c^T delta_c
            // Every iteration commits, with or without MMAs: after a failure the commits
            // still pace the chain one generation at a time.
            for (int c = 0; c < nchunks; ++c) {
                named_bar_sync(kNamedIssue, kIssueCount);
                const bool live = !*k2fail;
                tc_fence_after();
                if (elect_one()) {
                    if (live)
                        mma_ts(tmem + kColS, tmem + kColDA + 8u * (c & 1), sdesc(stage(c) + kB2, kLbo, kSboB2),
                               idesc128, 1);
                    // Mq_c delta_c into chunk c's output partial (MMA1(c) wrote it; the chain
                    // reads it after this commit), kept off the MMA1 issuers' path.
                    if (live && with_out)
                        mma_ts(tmem + kColD1 + kD1Buf * (c & 1) + 16, tmem + kColDA + 8u * (c & 1),
                               sdesc(stage(c) + kB3, kLbo, kSboB3), idesc16, 1);
                    tc_commit(bar(BAR_SDONE));
                }
                __syncwarp();
                // Chunk c-1's stage is no longer read (its last MMAs completed before the
                // chain reached this point): hand it back to the K1 CTA.
                if (live && c > 0 && lane == 0)
                    mbar_arrive_remote_relaxed(mapa(bar(BAR_OUT_FREE + (c - 1) % kRecvStages), 0));
            }
        } else if (warp == kMma1WarpA || warp == kMma1WarpB) {
            // ---- after EMIT(c): warp 10 issues MMA1(c+1) over keys 0-63 plus the lookahead
            // term (the output term Mq_c delta_c goes with the state update); warp 9 issues
            // MMA1(c+1) over keys 64-127 and then the output tile's TMA store.  Each commits
            // to BAR_D1 once per EMIT generation (phase c+1), with or without MMAs (see
            // warp 11).
            const int kh = warp == kMma1WarpA ? 0 : 1;
            const int tile_head = out_head();  // once: the tile stores below run every chunk
            auto mma1 = [&](int c) {
                const uint32_t d = tmem + kColD1 + kD1Buf * (c & 1) + 32u * kh;
                const uint32_t b1 = stage(c) + kB1;
#pragma unroll
                for (int s4 = 0; s4 < 4; ++s4) {
                    const int kk = 4 * kh + s4;
                    mma_ts(d, tmem + kColSA + 8u * kk, sdesc(b1 + kk * 2 * kLbo, kLbo, kSboB1), idesc1, s4);
                }
                if (kh == 0 && c > 0)
                    mma_ts(d, tmem + kColDA + 8u * ((c - 1) & 1),
                           sdesc(sbase + kSmPR + ((c - 1) % kPRSlots) * kPRBytes, kLbo, kSboB3), idesc1, 1);
            };
            // EMIT(-1): S_0 and its bf16 copy written
            named_bar_sync(kNamedEmit, kEmitCount);
            if (nchunks > 0) {
                const bool live = !*k2fail && __all_sync(0xffffffffu, landed_or_wait(0));
                if (!live && lane == 0) *k2fail = 1;
                tc_fence_after();
                if (elect_one()) {
                    if (live) mma1(0);
                    tc_commit(bar(BAR_D1));
                }
                __syncwarp();
            }
            for (int c = 0; c < nchunks; ++c) {
                const bool has_next = c + 1 < nchunks;
                // Operands of MMA1(c+1) are checked before the barrier: they do not
                // depend on it, and the MMAs then go out right after it.
                bool pre = true;
                if (has_next && !*k2fail) {
                    pre = landed_or_wait(c + 1);
                    if (kh == 0)
                        pre = pre && (ld_acquire_cta(pr_ready) > c ||
                                      mbar_wait(bar(BAR_PR_FULL + c % kPRSlots), (c / kPRSlots) & 1, lim));
                }
                named_bar_sync(kNamedEmit, kEmitCount);  // EMIT(c)
                bool live = !*k2fail && __all_sync(0xffffffffu, pre);
                if (!live && lane == 0) *k2fail = 1;
                tc_fence_after();
                if (elect_one()) {
                    if (live && has_next) mma1(c + 1);
                    tc_commit(bar(BAR_D1));
                }
                __syncwarp();
                if (live && kh == 1 && c > 0 && with_out && lane == 0) {
                    // Output tile of chunk c-1 (written by the chain before EMIT(c)).  The
                    // chain refills this warp's tiles only after D1 phases this warp
                    // commits later, so the drain below (all but the two newest stores)
                    // covers the store of the chunk four back, whose tile comes next.
                    const int32_t t0p = (int32_t)(bos + (int64_t)(c - 1) * kChunk);
                    tma_store_3d(&tm_out, sbase + kSmOTile + ((c - 1) % kOTiles) * kOTileBytes, 0, tile_head, t0p);
                    bulk_commit();
                    bulk_wait_read<2>();
                }
                __syncwarp();
            }
            if (kh == 1 && lane == 0) bulk_wait0();  // TMA stores complete before exit
        } else {
            // ---- state chain (warps 1-8, 256 threads)
            const int quad = warp & 3;                 // TMEM lane quadrant = SM sub-partition
            const int hf = (warp - 1) >> 2;            // key columns 64hf.., delta rows 8hf..
            const int j = 32 * quad + lane;            // value column owned by this thread
            const uint32_t lanes = (uint32_t)(32 * quad) << 16;
            const uint32_t tS = tmem + lanes + kColS + 64u * hf;
            const uint32_t tSA = tmem + lanes + kColSA + 32u * hf;
            // State rows: initial state at this CTA's row; final state at its row, or (segment
            // runs) at sequence b for the last segment only.
            const size_t soff = ((size_t)n * p.H + h) * kD * kD;
            size_t foff = soff;
            bool write_final = p.sfin != nullptr && (!kGrouped || head_map(out_head(), p.H, p.Hq).state_owner);
            if (p.flags & kFlagFinalLastSeg) {
                write_final = write_final && seg_id == seg_count - 1;
                foff = ((size_t)seq_id * p.H + h) * kD * kD;
            }
            uint32_t sreg[64];
            // Initial state S0[i][j] for keys i of this half -> S^T[j][i], and its bf16 copy.
            if (p.flags & kFlagIdentityS0) {
#pragma unroll
                for (int i = 0; i < 64; ++i) sreg[i] = (64 * hf + i == j) ? __float_as_uint(1.f) : 0u;
            } else if (p.s0 == nullptr) {
#pragma unroll
                for (int i = 0; i < 64; ++i) sreg[i] = 0u;
            } else if (p.s0_bf16) {  // bf16 states: widened exactly
                const __nv_bfloat16* s0h = static_cast<const __nv_bfloat16*>(p.s0);
#pragma unroll
                for (int i = 0; i < 64; ++i)
                    sreg[i] = __float_as_uint(__bfloat162float(s0h[soff + (size_t)(64 * hf + i) * kD + j]));
            } else {
                const float* s0f = static_cast<const float*>(p.s0);
#pragma unroll
                for (int i = 0; i < 64; ++i) sreg[i] = __float_as_uint(s0f[soff + (size_t)(64 * hf + i) * kD + j]);
            }
            tmem_st32(tS, sreg);
            tmem_st32(tS + 32, sreg + 32);
            {
                uint32_t pk[32];
#pragma unroll
                for (int i = 0; i < 32; ++i)
                    pk[i] = pack_bf16(__uint_as_float(sreg[2 * i]), __uint_as_float(sreg[2 * i + 1]));
                tmem_st32(tSA, pk);
            }
            tmem_wait_st();
            tc_fence_before();
            // Arrive on an issuer barrier.  After a failure the waits that pace the chain
            // are skipped, so the chain then waits at the barrier too and can never be a
            // generation ahead of the issuers.
            auto chain_arrive = [&](uint32_t id, uint32_t count) {
                if (*k2fail) named_bar_sync(id, count);
                else named_bar_arrive(id, count);
            };
            chain_arrive(kNamedEmit, kEmitCount);  // EMIT(-1)
            // Sum of the two K-half partials of 8 accumulator columns (rows 8hf..8hf+7);
            // `col` selects the W (0) or the output (16) half of each partial.
            auto ld_partials = [&](int buf, uint32_t col, float (&v)[8]) {
                uint32_t a[8], b[8];
                const uint32_t base = tmem + lanes + kColD1 + kD1Buf * (uint32_t)buf + col + 8 * hf;
                tmem_ld8(base, a);
                tmem_ld8(base + 32, b);
                tmem_wait_ld_regs<8>(a);
                tmem_wait_ld_regs<8>(b);
#pragma unroll
                for (int r = 0; r < 8; ++r) v[r] = __uint_as_float(a[r]) + __uint_as_float(b[r]);
            };
            // Output rows 8hf.. of chunk cp: through an output tile (stored by warp 9), or
            // with plain stores (the last chunk of the sequence, possibly ragged).
            auto emit_out = [&](int cp, bool tile_ok) {
                const int64_t t0p = bos + (int64_t)cp * kChunk;
                const int Cp = (eos - t0p < kChunk) ? (int)(eos - t0p) : kChunk;
                float o[8];
                ld_partials(cp & 1, 16, o);
                if (tile_ok) {
                    __nv_bfloat16* tile =
                        reinterpret_cast<__nv_bfloat16*>(smem + kSmOTile + (cp % kOTiles) * kOTileBytes);
#pragma unroll
                    for (int r = 0; r < 8; ++r) tile[(8 * hf + r) * kD + j] = __float2bfloat16_rn(p.scale * o[r]);
                } else {
#pragma unroll
                    for (int r = 0; r < 8; ++r) {
                        const int row = 8 * hf + r;
                        if (row < Cp)
                            p.out[((t0p + row) * out_heads() + out_head()) * kD + j] =
                                __float2bfloat16_rn(p.scale * o[r]);
                    }
                }
            };
            for (int c = 0; c < nchunks; ++c) {
                const bool has_next = c + 1 < nchunks;
                const int ks = c % kRecvStages;
                // The SDONE and D1 waits pace the chain against the issuers and are taken
                // even after a failure (the issuers then commit without MMAs).
                bool w = !*k2fail && landed_or_wait(c);                    // U_c, exp(gam_C(c))
                if (c > 0 && !mbar_wait_now(bar(BAR_SDONE), (c - 1) & 1, lim)) w = false;  // S_c complete
                uint32_t pk[32];  // bf16 copy of D_{c+1}, written once MMA1(c) has read D_c
                if (w) {
                    tc_fence_after();
                    // D_{c+1} = Diag(exp gam_C(c)) S_c, in place: warp 11 then adds Kbar_c^T delta_c.
                    tmem_ld32(tS, sreg);
                    tmem_ld32(tS + 32, sreg + 32);
                    tmem_wait_ld_regs<64>(sreg);
                    const float4* gc4 = reinterpret_cast<const float4*>(smem + kSmRecv + ks * kOutBytes + kGC) + 16 * hf;
#pragma unroll
                    for (int i4 = 0; i4 < 16; ++i4) {
                        const float4 gv = gc4[i4];
                        float a = __uint_as_float(sreg[4 * i4]), b = __uint_as_float(sreg[4 * i4 + 1]);
                        float cc = __uint_as_float(sreg[4 * i4 + 2]), d = __uint_as_float(sreg[4 * i4 + 3]);
                        mul2(a, b, gv.x, gv.y);
                        mul2(cc, d, gv.z, gv.w);
                        sreg[4 * i4] = __float_as_uint(a);
                        sreg[4 * i4 + 1] = __float_as_uint(b);
                        sreg[4 * i4 + 2] = __float_as_uint(cc);
                        sreg[4 * i4 + 3] = __float_as_uint(d);
                    }
                    tmem_st32(tS, sreg);
                    tmem_st32(tS + 32, sreg + 32);
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        pk[i] = pack_bf16(__uint_as_float(sreg[2 * i]), __uint_as_float(sreg[2 * i + 1]));
                }
                if (!mbar_wait_now(bar(BAR_D1), c & 1, lim)) w = false;
                {
                    if (w) {
                        tc_fence_after();
                        // MMA1(c) has read D_c and [P_{c-1} ; R_{c-1}]: overwrite / hand back.
                        if (warp == 8 && lane == 0 && c > 0) {
                            mbar_arrive(bar(BAR_PR_FREE + (c - 1) % kPRSlots));
                            st_release_cta(pr_used, c);  // operands 0 .. c-1 read
                        }
                        if (has_next) tmem_st32(tSA, pk);
                        // delta^T = U^T - (W D + P delta_prev)^T for rows 8hf .. 8hf+7
                        float dsum[8];
                        ld_partials(c & 1, 0, dsum);
                        const float* U = reinterpret_cast<const float*>(smem + kSmRecv + ks * kOutBytes + kU);
                        uint32_t pk4[4];
#pragma unroll
                        for (int r = 0; r < 4; ++r) {
                            const int r0 = 8 * hf + 2 * r;
                            pk4[r] = pack_bf16(U[r0 * kURow + j] - dsum[2 * r], U[(r0 + 1) * kURow + j] - dsum[2 * r + 1]);
                        }
                        tmem_st4(tmem + lanes + kColDA + 8u * (c & 1) + 4u * hf, pk4);
                    }
                }
                if (!w) *k2fail = 1;
                tmem_wait_st();
                tc_fence_before();
                chain_arrive(kNamedIssue, kIssueCount);  // ISSUE(c)
                // Output of chunk c-1 (its Mq delta term completed with D1(c)), while the
                // state update runs; the last chunk's output follows the loop.
                if (w && c > 0 && with_out) emit_out(c - 1, true);
                fence_proxy_async_smem();
                tc_fence_before();
                chain_arrive(kNamedEmit, kEmitCount);  // EMIT(c)
            }
            // Output of the last chunk (its Mq delta term commits to D1 phase nchunks) and
            // the final state.
            const bool fin = !*k2fail && nchunks > 0 && mbar_wait(bar(BAR_SDONE), (nchunks - 1) & 1, lim) &&
                             mbar_wait(bar(BAR_D1), nchunks & 1, lim);
            if (fin) {
                tc_fence_after();
                if (with_out) emit_out(nchunks - 1, false);
            }
            if (!*k2fail && write_final) {
                tc_fence_after();
                tmem_ld32(tS, sreg);
                tmem_ld32(tS + 32, sreg + 32);
                tmem_wait_ld_regs<64>(sreg);
                if (p.sfin_bf16) {  // bf16 states: rounded to nearest even
                    __nv_bfloat16* fh = static_cast<__nv_bfloat16*>(p.sfin);
#pragma unroll
                    for (int i = 0; i < 64; ++i)
                        fh[foff + (size_t)(64 * hf + i) * kD + j] = __float2bfloat16_rn(__uint_as_float(sreg[i]));
                } else {
                    float* ff = static_cast<float*>(p.sfin);
#pragma unroll
                    for (int i = 0; i < 64; ++i) ff[foff + (size_t)(64 * hf + i) * kD + j] = __uint_as_float(sreg[i]);
                }
            } else if (nchunks > 0 && !fin) {
                *k2fail = 1;
            }
            tmem_wait_st();
            tmem_wait_ld();
        }
        // Every MMA the three issuers started completes before TMEM is released.
        if (warp == kMma1WarpA || warp == kMma1WarpB || warp == kUpdateWarp) {
            if (elect_one()) tc_commit(bar(BAR_DRAIN));
            __syncwarp();
            if (!mbar_wait(bar(BAR_DRAIN), 0, kDrainLimit) && lane == 0) record(p.status, kStatusTimeout);
        }
        if (*k2fail && lane == 0) record(p.status, kStatusTimeout);
    }

    tc_fence_before();
    cluster_sync();  // neither CTA leaves while its peer may still access its memory
    if (rank == 1 && warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem_base, kTmemCols);
    }
}

}  // namespace

size_t serial_smem_bytes() { return kSmemBytes; }
int serial_block_threads() { return kThreads; }
const void* serial_kernel_symbol() { return reinterpret_cast<const void*>(&kda_fwd_tc_kernel<false>); }
const void* grouped_kernel_symbol() { return reinterpret_cast<const void*>(&kda_fwd_tc_kernel<true>); }

cudaError_t launch_serial(const FwdParams& p, const TensorMaps& maps, cudaStream_t stream) {
    const long long rows = p.seg_len > 0 ? (p.cu ? (long long)p.rows : (long long)p.N * p.nseg_used)
                                         : (long long)p.N;
    const long long clusters = rows * (p.Hq > p.H ? p.Hq : p.H);
    if (clusters == 0) return cudaSuccess;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(2 * clusters), 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (p.Hq != p.H)
        return cudaLaunchKernelEx(&cfg, kda_fwd_tc_kernel<true>, maps.q, maps.k, maps.v, maps.g,
                                  maps.out, p);
    return cudaLaunchKernelEx(&cfg, kda_fwd_tc_kernel<false>, maps.q, maps.k, maps.v, maps.g,
                              maps.out, p);
}

}  // namespace kda
