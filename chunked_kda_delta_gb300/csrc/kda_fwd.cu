// kda_fwd.cu -- KDA forward prefill for sm_103a: one 2-CTA thread-block cluster per
// (sequence, head) chain; the state is advanced 32 tokens (two 16-token chunks) per step,
// held in tensor memory (TMEM) for the whole sequence; every dense contraction runs on
// tcgen05 with operands staged in shared memory by TMA or by the CUDA cores.
//
// The method (cuLA PR #103 "feat(kda/sm90): FlashKDA prefill port + intracard-CP
// prefill", commit notes): chunks of 16 tokens, head size 128, forward only; K1 builds
// the decayed q/k, applies beta and forms the WY inverse of each chunk by a 16x16
// unit-lower-triangular solve; K2 carries the state from chunk to chunk and forms the
// output.  For a step of C <= 32 rows (two chunks) with step-start state S (Dk x Dv),
// step-cumulative log-decay gam_r = sum_{m<=r} g_m (per channel):
//   A    = strict_lower(beta_r (Kt Kh^T)_rs),  Kt = K o e^{gam},  Kh = K o e^{-gam}
//   T    = (I + A)^{-1}: the two chunks' 16x16 inverses (diagonal blocks) and their
//          cross block (block forward substitution), Tb = T diag(beta)
//   W    = Tb Kt,  U = Tb V,  Mq = lower(Qt Kh^T),  Qt = Q o e^{gam}
//   delta = U - W S,  O = scale (Qt S + Mq delta)
//   S   <- Diag(e^{gam_C}) S + Kb^T delta,  Kb = K o e^{gam_C - gam}
// Kt, Qt, Kb and e^{gam_C} never exceed 1 for g <= 0; Kh grows up to e^{-gam_C}, which
// stays inside the fp32 / bf16 range while a step's total log-decay is above -80 per
// channel (the kernel records KDA_ERR_UNSUPPORTED_DECAY-free: steps beyond it are
// computed by the exact pairwise path, see k1_slow_grams).
//
// One-step lookahead in K2: with D_p = Diag(e^{gam_C(p-1)}) S_{p-1},
//   W_p S_p = W_p D_p + P_{p-1} delta_{p-1},  P_{p-1} = W_p Kb_{p-1}^T  (Qt, R alike),
// so the big product of step p with the state (MMA1, K = 128) runs on D_p and only a
// K = 32 product with delta_{p-1} sits on the chain.  U enters the same accumulator
// through Vt (-Tb)^T (the negate-B bit), so delta_p^T = -(accumulator).
//
// Work split.  CTA rank 0 ("K1"): TMA producer (q, k, g), eight elementwise warps
// (decayed operands), a Gram issuer ([Kt; Qt] x [Kh; Kb_prev]^T, one M=128 N=64 group),
// two solve warps (Tb and P = Tb (beta o X), X = Kt Kb_prev^T), a W issuer
// (W^T = Kt^T Tb^T), four TMEM epilogue warps and a shipper that bulk-copies each step's
// W, Tb, Mq and [P; R] (16 KB) into the K2 CTA.  CTA rank 1 ("K2"): its own TMA producer
// (q, k, v, g: it forms Qt, Kb and the V operand itself, so only 16 KB per step cross
// the cluster), four warps building those, four delta warps (delta, the lookahead and
// U products, the output), four decay warps (the state's decay in place, its bf16 copy,
// the state update), two MMA1 issuers and a relay that tells K1 when a copy landed.
// Every wait is bounded; on exhaustion the kernel records KDA_ERR_DEVICE_TIMEOUT, tells
// the peer CTA, drains its in-flight copies and MMAs and exits.
#include <cuda.h>

#include "kda_internal.cuh"
#include "kda_ptx.cuh"

// Timeline hooks for profiling builds (compiled with KDA_TRACE_POINT defined); no code
// otherwise.
#ifndef KDA_TRACE_POINT
#define KDA_TRACE_POINT(ev, st)
#endif

namespace kda {
namespace {

using namespace ptx;

constexpr int kBlk = 32;  // tokens per chain step
constexpr int kThreads = 512;
constexpr int64_t kDrainLimit = 1ll << 24;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kFastLimit = 80.f;  // nats of decay per step for the factored Grams

// ---------------------------------------------------------------- layouts
// Tiles of R rows x 128 channels (bf16): 16 bytes hold 8 consecutive rows of one
// channel; row group a (rows 8a..8a+7) starts at a * kRG.  As an MMA operand with rows
// along M/N and channels along K it is MN-major (LBO 128 = next 8 channels, SBO 2048 =
// next 8 rows); with channels along M/N and rows along K it is K-major (LBO 2048, SBO 128).
constexpr uint32_t kRG = 2048;
__device__ __forceinline__ uint32_t tile_off(int r, int c) {
    return (uint32_t)(r >> 3) * kRG + (uint32_t)c * 16u + (uint32_t)(r & 7) * 2u;
}
// 32 x 32 (or 64 x 32) bf16 matrices [n][s] with n along N and s along K.
// Tb, MN-major (n contiguous): LBO 128 (next 8 s), SBO 512 (next 8 n).
__device__ __forceinline__ uint32_t tb_off(int n, int s) {
    return (uint32_t)(s >> 3) * 128u + (uint32_t)(n >> 3) * 512u + (uint32_t)(s & 7) * 16u + (uint32_t)(n & 7) * 2u;
}
// Mq and [P; R], K-major (s contiguous): LBO 128 (next 8 s), SBO 512 (next 8 n).
__device__ __forceinline__ uint32_t km_off(int n, int s) {
    return (uint32_t)(n >> 3) * 512u + (uint32_t)(s >> 3) * 128u + (uint32_t)(n & 7) * 16u + (uint32_t)(s & 7) * 2u;
}

// ---------------------------------------------------------------- shared memory maps
// K1 CTA
constexpr int K1_IN = 0;  // 2 stages: q | k | g | beta
constexpr int K1_IN_STAGE = 33792, K1_IN_Q = 0, K1_IN_K = 8192, K1_IN_G = 16384, K1_IN_BETA = 32768;
constexpr int K1_A = K1_IN + 2 * K1_IN_STAGE;  // 2 Gram-A areas [Kt; Qt] (64 rows)
constexpr int K1_A_BYTES = 16384;
constexpr int K1_B = K1_A + 2 * K1_A_BYTES;    // 3 Gram-B areas [Kh; Kb_prev] (64 rows)
constexpr int K1_B_BYTES = 16384;
constexpr int K1_OUT = K1_B + 3 * K1_B_BYTES;  // 3 out stages: W | Tb | Mq | PR
constexpr int OUT_W = 0, OUT_TB = 8192, OUT_MQ = 10240, OUT_PR = 12288, OUT_BYTES = 16384;
constexpr int kOutStages = 3;
constexpr int K1_AS = K1_OUT + kOutStages * OUT_BYTES;  // A (transposed, fp32 32x32)
constexpr int K1_XS = K1_AS + 4096;            // beta o X (fp32, column c at c * 36)
constexpr int K1_BETA = K1_XS + 32 * 36 * 4;   // beta of the step being solved, [2][32]
constexpr int K1_SCAN = K1_BETA + 256;         // elementwise scan, [4][64] float4
constexpr int K1_END = K1_SCAN + 4096;
// K2 CTA
constexpr int K2_IN = 0;  // 2 stages: q | k | v | g
constexpr int K2_IN_STAGE = 40960, K2_IN_Q = 0, K2_IN_K = 8192, K2_IN_V = 16384, K2_IN_G = 24576;
constexpr int K2_RECV = K2_IN + 2 * K2_IN_STAGE;  // 3 stages
constexpr int RV_W = 0, RV_QT = 8192, RV_KB = 16384, RV_V = 24576, RV_TB = 32768, RV_MQ = 34816,
              RV_PR = 36864, RV_GC = 40960, RV_STAGE = 41984;
static_assert(RV_QT == RV_W + 8192, "Qt follows W: rows 32..63 of the MMA1 operand");
constexpr int K2_OTILE = K2_RECV + 3 * RV_STAGE;  // 2 output tiles [32][128] bf16
constexpr int K2_SCAN = K2_OTILE + 2 * 8192;      // [2][64] float4
constexpr int K2_END = K2_SCAN + 2048;
// Barriers and flags (same offset in both CTAs, so a peer's barrier is mapa(local, peer)).
constexpr int kSmBar = (K2_END > K1_END ? K2_END : K1_END);
constexpr int kNumBars = 48;
constexpr int kSmFail = kSmBar + kNumBars * 8;   // int32: this CTA gave up
constexpr int kSmSlow = kSmFail + 4;             // int32 [2]: K1 step used the exact Gram path
constexpr int kSmTmem = kSmSlow + 8;             // TMEM base address
constexpr int kSmemBytes = kSmTmem + 8;
static_assert(kSmemBytes <= 232448, "shared memory");
static_assert(K1_IN + K1_IN_STAGE * 2 <= K1_A && K1_A % 1024 == 0 && K1_B % 1024 == 0, "K1 map");
static_assert(K2_RECV % 1024 == 0 && RV_STAGE % 1024 == 0 && K2_OTILE % 1024 == 0, "K2 map");
static_assert(RV_TB + 8192 == RV_GC && OUT_TB + 8192 == OUT_BYTES, "Tb | Mq | PR ship as one copy");

enum {  // K1 barriers
    B1_IN_FULL = 0, B1_IN_EMPTY = 2, B1_EDONE = 4, B1_GDONE = 6, B1_GREAD = 8, B1_TBREADY = 10,
    B1_WDONE = 12, B1_OUTREADY = 14, B1_RECVFREE = 18 /* 3 */, B1_DRAIN = 21,
    B1_OUTFREE = 43 /* 3 */
};
enum {  // K2 barriers
    B2_IN_FULL = 0, B2_IN_EMPTY = 2, B2_RECVFULL = 24 /* 3 */, B2_LOCALREADY = 27 /* 3 */,
    B2_LOCALFREE = 30 /* 3 */, B2_L = 33, B2_MMA1 = 34, B2_LOOK = 35, B2_SAREADY = 36 /* 2 */,
    B2_SDONE = 38 /* 2 */, B2_DELTA = 40, B2_DRAIN = 41, B2_NEVER = 42
};
static_assert(B2_NEVER < kNumBars && B1_OUTFREE + 3 <= kNumBars, "barriers");
// Named barriers (ids 1..15; ids are per CTA)
constexpr uint32_t NB_E = 1, NB_SOLVE = 2, NB_EPI = 3, NB_DELTA = 4, NB_DECAY = 5, NB_ELITE = 6;

// TMEM columns
constexpr uint32_t K1_TM_G = 0, K1_TM_W = 128, K1_TM_COLS = 256;
constexpr uint32_t K2_TM_S = 0, K2_TM_SA = 128, K2_TM_ACC = 256, K2_TM_DA = 448, K2_TM_COLS = 512;

__device__ __forceinline__ void record(int32_t* status, int32_t code) { atomicCAS(status, kStatusOk, code); }

// Bounded wait that also gives up as soon as this CTA has failed elsewhere.  The thread
// sleeps in hardware between checks (up to kWaitNs per round, woken when the phase
// completes), so waiting warps leave the issue slots to the warps doing the work.  `lim`
// counts polling iterations as elsewhere in the library; one suspended round stands for
// kRoundIters of them, which bounds a wait that never completes to about
// lim / kRoundIters * kWaitNs (0.16 s at the default limit).
constexpr uint32_t kWaitNs = 10000;
constexpr int64_t kRoundIters = 256;
__device__ __forceinline__ bool bwait(uint32_t bar, uint32_t parity, int64_t lim, const volatile int32_t* fail) {
    if (mbar_try_wait(bar, parity)) return true;
    for (int64_t i = 0; i < lim; i += kRoundIters) {
        if (mbar_try_wait_ns(bar, parity, kWaitNs)) return true;
        if (*fail) return false;
    }
    return false;
}
__device__ __forceinline__ bool bwait_cluster(uint32_t bar, uint32_t parity, int64_t lim,
                                              const volatile int32_t* fail) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    for (int64_t i = 0; i < lim; i += kRoundIters) {
        if (mbar_try_wait_cluster_ns(bar, parity, kWaitNs)) return true;
        if (*fail) return false;
    }
    return false;
}

// ---------------------------------------------------------------- elementwise stage
// Decayed operands of one step for channels 2pc, 2pc+1 and rows [part * R, part * R + R),
// R = 32 / kParts; kParts * 64 threads take part, meeting once at named barrier `nb`.
// Writes (null pointers are skipped): kt = K o e^{gam}, qt = Q o e^{gam}, kb = K o
// e^{gam_C - gam}, kh = Kb o e^{-gam_C} (= K o e^{-gam}, the factor clamped to 2^126),
// vt = V (zero when zero_v) into tiles of the layout above (row offset `*_row0`), and
// e^{gam_C} into gc[128].  Returns true when a channel's step log-decay is below
// -kFastLimit (the factored Grams are then replaced by the exact ones).
struct ETiles {
    unsigned char *kt, *qt, *kb, *kh, *vt;
    int kt_row0, qt_row0, kb_row0, kh_row0;
    float* gc;
};
template <int kParts>
__device__ __forceinline__ bool e_step(const unsigned char* in_q, const unsigned char* in_k,
                                       const unsigned char* in_v, const float* in_g, int C, int part, int pc,
                                       float4* scan, uint32_t nb, const ETiles& o, bool zero_v) {
    constexpr int R = kBlk / kParts;
    const int r0 = part * R;
    const float2 l2e = make_float2(kLog2e, kLog2e);
    float2 e[R];
    float2 sum = make_float2(0.f, 0.f), prod = make_float2(1.f, 1.f);
#pragma unroll
    for (int i = 0; i < R; ++i) {
        const int r = r0 + i;
        const float2 gv = r < C ? reinterpret_cast<const float2*>(in_g)[r * 64 + pc] : make_float2(0.f, 0.f);
        sum = add2(sum, gv);
        e[i] = ex2x2(mul2f(gv, l2e));
        prod = mul2f(prod, e[i]);
    }
    scan[part * 64 + pc] = make_float4(sum.x, sum.y, prod.x, prod.y);
    named_bar_sync(nb, kParts * 64);
    float2 pre = make_float2(1.f, 1.f), post = make_float2(1.f, 1.f), tot = make_float2(0.f, 0.f);
#pragma unroll
    for (int q = 0; q < kParts; ++q) {
        const float4 s = scan[q * 64 + pc];
        tot = add2(tot, make_float2(s.x, s.y));
        if (q < part) pre = mul2f(pre, make_float2(s.z, s.w));
        if (q > part) post = mul2f(post, make_float2(s.z, s.w));
    }
    const bool slow = tot.x < -kFastLimit || tot.y < -kFastLimit;
    // e^{-gam_C}, its exponent clamped so that Kh stays finite (slow steps ignore Kh)
    const float2 inv = ex2x2(make_float2(fminf(-tot.x * kLog2e, 126.f), fminf(-tot.y * kLog2e, 126.f)));
    if (o.gc != nullptr && part == 0) reinterpret_cast<float2*>(o.gc)[pc] = ex2x2(mul2f(tot, l2e));
    // suffix products e^{gam_C - gam_r} = post * prod_{m > r, m in part} e_m
    float2 sfx[R];
    {
        float2 s = post;
#pragma unroll
        for (int i = R - 1; i >= 0; --i) {
            sfx[i] = s;
            s = mul2f(s, e[i]);
        }
    }
    const uint32_t* q2 = reinterpret_cast<const uint32_t*>(in_q);
    const uint32_t* k2 = reinterpret_cast<const uint32_t*>(in_k);
    const uint32_t* v2 = reinterpret_cast<const uint32_t*>(in_v);
    float2 pf = pre;
    const int c0 = 2 * pc, c1 = 2 * pc + 1;
#pragma unroll
    for (int grp = 0; grp < R / 8; ++grp) {
        uint32_t kt0[4], kt1[4], qt0[4], qt1[4], kb0[4], kb1[4], kh0[4], kh1[4], v0[4], v1[4];
#pragma unroll
        for (int h = 0; h < 4; ++h) {
            float2 ktv[2], qtv[2], kbv[2], khv[2];
            uint32_t vv[2];
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const int i = grp * 8 + 2 * h + u, r = r0 + i;
                const bool valid = r < C;
                pf = mul2f(pf, e[i]);  // e^{gam_r}
                const uint32_t kv = valid ? k2[r * 64 + pc] : 0u;
                const uint32_t qv = (valid && o.qt) ? q2[r * 64 + pc] : 0u;
                vv[u] = (valid && o.vt && !zero_v) ? v2[r * 64 + pc] : 0u;
                const float2 kf = bf2_to_f2(kv), qf = bf2_to_f2(qv);
                ktv[u] = mul2f(kf, pf);
                qtv[u] = mul2f(qf, pf);
                kbv[u] = mul2f(kf, sfx[i]);
                khv[u] = mul2f(kbv[u], inv);
            }
            kt0[h] = pack_bf16(ktv[0].x, ktv[1].x);
            kt1[h] = pack_bf16(ktv[0].y, ktv[1].y);
            qt0[h] = pack_bf16(qtv[0].x, qtv[1].x);
            qt1[h] = pack_bf16(qtv[0].y, qtv[1].y);
            kb0[h] = pack_bf16(kbv[0].x, kbv[1].x);
            kb1[h] = pack_bf16(kbv[0].y, kbv[1].y);
            kh0[h] = pack_bf16(khv[0].x, khv[1].x);
            kh1[h] = pack_bf16(khv[0].y, khv[1].y);
            v0[h] = (vv[0] & 0xffffu) | (vv[1] << 16);
            v1[h] = (vv[0] >> 16) | (vv[1] & 0xffff0000u);
        }
        const int r = r0 + grp * 8;
        auto put = [&](unsigned char* t, int row0, const uint32_t (&a)[4], const uint32_t (&b)[4]) {
            if (t == nullptr) return;
            *reinterpret_cast<uint4*>(t + tile_off(row0 + r, c0)) = make_uint4(a[0], a[1], a[2], a[3]);
            *reinterpret_cast<uint4*>(t + tile_off(row0 + r, c1)) = make_uint4(b[0], b[1], b[2], b[3]);
        };
        put(o.kt, o.kt_row0, kt0, kt1);
        put(o.qt, o.qt_row0, qt0, qt1);
        put(o.kb, o.kb_row0, kb0, kb1);
        put(o.kh, o.kh_row0, kh0, kh1);
        put(o.vt, 0, v0, v1);
    }
    return slow;
}

// ---------------------------------------------------------------- exact Grams (strong decay)
// A (transposed, beta-scaled, strict lower) and Mq (bf16 K-major) of a step computed pair by
// pair with e^{gam_r - gam_s} formed directly, so no factor exceeds 1 for g <= 0.  Run by
// the 64 threads of the two solve warps from the step's inputs (kept until it is done).
__device__ void k1_slow_grams(const unsigned char* in, int C, int t, float* As, const float* beta,
                              unsigned char* mq) {
    const __nv_bfloat16* q = reinterpret_cast<const __nv_bfloat16*>(in + K1_IN_Q);
    const __nv_bfloat16* k = reinterpret_cast<const __nv_bfloat16*>(in + K1_IN_K);
    const float* g = reinterpret_cast<const float*>(in + K1_IN_G);
    // pairs (r, s), s <= r < 32: 528; thread t takes pairs t, t + 64, ...
    for (int pidx = t; pidx < 528; pidx += 64) {
        int r = 0;
        while ((r + 1) * (r + 2) / 2 <= pidx) ++r;
        const int s = pidx - r * (r + 1) / 2;
        float aq = 0.f, ak = 0.f;
        if (r < C && s < C) {
            for (int c = 0; c < 128; ++c) {
                float d = 0.f;  // gam_r - gam_s = sum of g over rows s+1 .. r
                for (int m = s + 1; m <= r; ++m) d += g[m * 128 + c];
                const float f = ex2(d * kLog2e);
                const float kk = __bfloat162float(k[s * 128 + c]) * f;
                ak = fmaf(__bfloat162float(k[r * 128 + c]), kk, ak);
                aq = fmaf(__bfloat162float(q[r * 128 + c]), kk, aq);
            }
        }
        if (s < r) As[s * 32 + r] = beta[r] * ak;
        else As[s * 32 + r] = 0.f;
        for (int ss = r + 1; ss < 32 && s == r; ++ss) As[ss * 32 + r] = 0.f;  // upper part of row r
        *reinterpret_cast<__nv_bfloat16*>(mq + km_off(r, s)) = __float2bfloat16_rn(aq);
        for (int ss = r + 1; ss < 32 && s == r; ++ss)
            *reinterpret_cast<__nv_bfloat16*>(mq + km_off(r, ss)) = __float2bfloat16_rn(0.f);
    }
}

// x <- (I + A)^{-1} x for one column x (32 rows): forward substitution with A read
// column by column (As[m * 32 + r] = A[r][m]).  Rows go in blocks of four: the 4x4
// diagonal block is solved (a three-deep chain), then its four columns update every row
// below with independent FMAs, so the loads of the next panel overlap the chain.  The two
// 16-row halves are the chunks' WY blocks; the substitution crosses between them.
__device__ __forceinline__ void solve32(const float* As, float (&x)[32]) {
#pragma unroll
    for (int m0 = 0; m0 < 32; m0 += 4) {
        // diagonal block: A[m0+i][m0+j], i > j
        const float4 c0 = *reinterpret_cast<const float4*>(As + (m0 + 0) * 32 + m0);
        const float4 c1 = *reinterpret_cast<const float4*>(As + (m0 + 1) * 32 + m0);
        const float4 c2 = *reinterpret_cast<const float4*>(As + (m0 + 2) * 32 + m0);
        x[m0 + 1] = fmaf(-c0.y, x[m0], x[m0 + 1]);
        x[m0 + 2] = fmaf(-c0.z, x[m0], x[m0 + 2]);
        x[m0 + 3] = fmaf(-c0.w, x[m0], x[m0 + 3]);
        x[m0 + 2] = fmaf(-c1.z, x[m0 + 1], x[m0 + 2]);
        x[m0 + 3] = fmaf(-c1.w, x[m0 + 1], x[m0 + 3]);
        x[m0 + 3] = fmaf(-c2.w, x[m0 + 2], x[m0 + 3]);
        const float x0 = x[m0], x1 = x[m0 + 1], x2 = x[m0 + 2], x3 = x[m0 + 3];
#pragma unroll
        for (int r4 = m0 / 4 + 1; r4 < 8; ++r4) {
            const float4 a0 = *reinterpret_cast<const float4*>(As + (m0 + 0) * 32 + 4 * r4);
            const float4 a1 = *reinterpret_cast<const float4*>(As + (m0 + 1) * 32 + 4 * r4);
            const float4 a2 = *reinterpret_cast<const float4*>(As + (m0 + 2) * 32 + 4 * r4);
            const float4 a3 = *reinterpret_cast<const float4*>(As + (m0 + 3) * 32 + 4 * r4);
            float y0 = x[4 * r4 + 0], y1 = x[4 * r4 + 1], y2 = x[4 * r4 + 2], y3 = x[4 * r4 + 3];
            y0 = fmaf(-a0.x, x0, y0); y1 = fmaf(-a0.y, x0, y1); y2 = fmaf(-a0.z, x0, y2); y3 = fmaf(-a0.w, x0, y3);
            y0 = fmaf(-a1.x, x1, y0); y1 = fmaf(-a1.y, x1, y1); y2 = fmaf(-a1.z, x1, y2); y3 = fmaf(-a1.w, x1, y3);
            y0 = fmaf(-a2.x, x2, y0); y1 = fmaf(-a2.y, x2, y1); y2 = fmaf(-a2.z, x2, y2); y3 = fmaf(-a2.w, x2, y3);
            y0 = fmaf(-a3.x, x3, y0); y1 = fmaf(-a3.y, x3, y1); y2 = fmaf(-a3.z, x3, y2); y3 = fmaf(-a3.w, x3, y3);
            x[4 * r4 + 0] = y0; x[4 * r4 + 1] = y1; x[4 * r4 + 2] = y2; x[4 * r4 + 3] = y3;
        }
    }
}

template <bool kGrouped>
__global__ void __launch_bounds__(kThreads, 1)
kda_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
               const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_g,
               const __grid_constant__ CUtensorMap tm_out, const FwdParams p) {
    extern __shared__ __align__(1024) unsigned char smem[];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t rank = cluster_ctarank();
    const int Ho = kGrouped ? (p.Hq > p.H ? p.Hq : p.H) : p.H;
    const int row = (int)((blockIdx.x >> 1) / Ho);
    const int ho = (int)((blockIdx.x >> 1) % Ho);  // output head of this cluster
    int hq = ho, hk = ho, h = ho;
    bool state_owner = true;
    if (kGrouped) {
        const HeadMap hm = head_map(ho, p.H, p.Hq);
        hq = hm.hq;
        hk = hm.hk;
        h = hm.hs;
        state_owner = hm.state_owner;
    }
    int64_t bos, eos;
    int seq_id, seg_id, seg_count;
    if (!seq_range(p, row, bos, eos, seq_id, seg_id, seg_count)) return;  // both CTAs return
    const int64_t H = p.H;
    const int nsteps = (int)((eos - bos + kBlk - 1) / kBlk);
    const int64_t lim = p.wait_limit;
    const uint32_t sbase = smem_u32(smem);
    auto bar = [&](int i) { return sbase + (uint32_t)kSmBar + 8u * (uint32_t)i; };
    volatile int32_t* fail = reinterpret_cast<volatile int32_t*>(smem + kSmFail);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kSmTmem);
    const bool with_out = (p.flags & kFlagNoOutput) == 0;
    const bool zero_v = (p.flags & kFlagZeroV) != 0;
    // Give up: record the timeout, mark this CTA and its peer failed.
    auto give_up = [&]() {
        record(p.status, kStatusTimeout);
        *fail = 1;
        st_cluster_u32(mapa(sbase + (uint32_t)kSmFail, rank ^ 1u), 1u);
    };
    auto step_rows = [&](int st) -> int {
        const int64_t t0 = bos + (int64_t)st * kBlk;
        return (eos - t0 < kBlk) ? (int)(eos - t0) : kBlk;
    };

    if (tid == 0) {
        if (rank == 0) {
            for (int i = 0; i < 2; ++i) {
                mbar_init(bar(B1_IN_FULL + i), 1);
                mbar_init(bar(B1_IN_EMPTY + i), 1);
                mbar_init(bar(B1_EDONE + i), 1);
                mbar_init(bar(B1_GDONE + i), 1);
                mbar_init(bar(B1_GREAD + i), 1);
                mbar_init(bar(B1_TBREADY + i), 1);
                mbar_init(bar(B1_WDONE + i), 1);
                mbar_init(bar(B1_OUTREADY + i), 1);
            }
            for (int i = 0; i < 3; ++i) {
                mbar_init(bar(B1_RECVFREE + i), 1);
                mbar_init(bar(B1_OUTFREE + i), 1);
            }
            mbar_init(bar(B1_DRAIN), 2);
        } else {
            for (int i = 0; i < 2; ++i) {
                mbar_init(bar(B2_IN_FULL + i), 1);
                mbar_init(bar(B2_IN_EMPTY + i), 1);
                mbar_init(bar(B2_SAREADY + i), 1);
                mbar_init(bar(B2_SDONE + i), 1);
            }
            for (int i = 0; i < 3; ++i) {
                mbar_init(bar(B2_RECVFULL + i), 1);
                mbar_init(bar(B2_LOCALREADY + i), 1);
                mbar_init(bar(B2_LOCALFREE + i), 1);
            }
            mbar_init(bar(B2_L), 1);
            mbar_init(bar(B2_MMA1), 2);
            mbar_init(bar(B2_LOOK), 1);
            mbar_init(bar(B2_DELTA), 1);
            mbar_init(bar(B2_DRAIN), 4);
            mbar_init(bar(B2_NEVER), 1);
        }
        *fail = 0;
        reinterpret_cast<volatile int32_t*>(smem + kSmSlow)[0] = 0;
        reinterpret_cast<volatile int32_t*>(smem + kSmSlow)[1] = 0;
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(smem_u32(tmem_slot), rank == 0 ? K1_TM_COLS : K2_TM_COLS);
        tmem_relinquish();
    }
    if (rank == 0 && warp >= 4 && warp < 12) {
        // Kb of "step -1" (rows 32..63 of Gram-B area 0) is zero: the first lookahead
        // operands then vanish.
        const int et = tid - 128;
        uint4* z = reinterpret_cast<uint4*>(smem + K1_B + 4 * kRG);
        for (int i = et; i < (4 * (int)kRG) / 16; i += 256) z[i] = make_uint4(0, 0, 0, 0);
        fence_proxy_async_smem();
    }
    tc_fence_before();
    cluster_sync();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (rank == 0) {
        // =============================================================== K1 CTA
        if (warp == 0) {
            // ---- TMA producer: q, k, g of each step; beta with plain loads (2-byte rows).
            int issued = 0;
            for (int st = 0; st < nsteps; ++st) {
                const int s = st & 1;
                bool ok = st < 2 || bwait(bar(B1_IN_EMPTY + s), ((st >> 1) - 1) & 1, lim, fail);
                if (__any_sync(0xffffffffu, !ok)) {
                    if (lane == 0 && !*fail) give_up();
                    break;
                }
                unsigned char* in = smem + K1_IN + s * K1_IN_STAGE;
                const int64_t t = bos + (int64_t)st * kBlk + lane;
                reinterpret_cast<float*>(in + K1_IN_BETA)[lane] =
                    t < eos ? __bfloat162float(p.beta[t * H + h]) : 0.f;
                __syncwarp();
                if (lane == 0) {
                    const uint32_t dst = sbase + K1_IN + s * K1_IN_STAGE;
                    const int32_t t0 = (int32_t)(bos + (int64_t)st * kBlk);
                    mbar_arrive_expect_tx(bar(B1_IN_FULL + s), 32768u);
                    tma_load_3d(dst + K1_IN_Q, &tm_q, bar(B1_IN_FULL + s), 0, hq, t0);
                    tma_load_3d(dst + K1_IN_K, &tm_k, bar(B1_IN_FULL + s), 0, hk, t0);
                    tma_load_3d(dst + K1_IN_G, &tm_g, bar(B1_IN_FULL + s), 0, h, t0);
                    KDA_TRACE_POINT(0, st);
                }
                issued = st + 1;
            }
            if (lane == 0)
                for (int st = (issued >= 2 ? issued - 2 : 0); st < issued; ++st)
                    if (!mbar_wait(bar(B1_IN_FULL + (st & 1)), (st >> 1) & 1, kDrainLimit))
                        record(p.status, kStatusTimeout);
        } else if (warp == 1 || warp == 3) {
            // ---- MMA issuers: warp 1 the Grams, warp 3 W^T = Kt^T Tb^T.
            const bool gram = warp == 1;
            const uint32_t idg = idesc_bf16(128, 64) | kIdescAMn | kIdescBMn;
            const uint32_t idw = idesc_bf16(128, 32) | kIdescBMn;
            for (int st = 0; st < nsteps; ++st) {
                const int s = st & 1;
                bool ok;
                if (gram) {
                    ok = bwait(bar(B1_EDONE + s), (st >> 1) & 1, lim, fail) &&
                         (st < 2 || bwait(bar(B1_GREAD + s), ((st >> 1) - 1) & 1, lim, fail));
                } else {
                    ok = bwait(bar(B1_TBREADY + s), (st >> 1) & 1, lim, fail) &&
                         (st < 2 || bwait(bar(B1_OUTREADY + s), ((st >> 1) - 1) & 1, lim, fail));
                }
                if (__any_sync(0xffffffffu, !ok)) {
                    if (lane == 0 && !*fail) give_up();
                    break;
                }
                tc_fence_after();
                if (elect_one()) {
                    const uint32_t a = sbase + K1_A + s * K1_A_BYTES;
                    if (gram) {
                        const uint32_t b = sbase + K1_B + (st % 3) * K1_B_BYTES;
#pragma unroll
                        for (int kk = 0; kk < 8; ++kk)
                            mma_ss(tmem + K1_TM_G + 64u * s, sdesc(a + kk * 256, 128, kRG),
                                   sdesc(b + kk * 256, 128, kRG), idg, kk > 0);
                        tc_commit(bar(B1_GDONE + s));
                        KDA_TRACE_POINT(1, st);
                    } else {
                        const uint32_t tb = sbase + K1_OUT + (st % 3) * OUT_BYTES + OUT_TB;
#pragma unroll
                        for (int kk = 0; kk < 2; ++kk)
                            mma_ss(tmem + K1_TM_W + 32u * s, sdesc(a + kk * 2 * kRG, kRG, 128),
                                   sdesc(tb + kk * 256, 128, 512), idw, kk > 0);
                        tc_commit(bar(B1_WDONE + s));
                        KDA_TRACE_POINT(2, st);
                    }
                }
                __syncwarp();
            }
            if (elect_one()) tc_commit(bar(B1_DRAIN));
            __syncwarp();
            if (!mbar_wait(bar(B1_DRAIN), 0, kDrainLimit) && lane == 0) record(p.status, kStatusTimeout);
        } else if (warp == 2) {
            // ---- shipper: W | Tb | Mq | PR of each step into the K2 CTA's receive stage.
            int shipped = 0;
            if (lane == 0) {
                for (int st = 0; st < nsteps; ++st) {
                    const int s = st & 1, rs = st % 3;  // out stage st % 3 as well
                    bool ok = bwait(bar(B1_OUTREADY + s), (st >> 1) & 1, lim, fail) &&
                              (st < 3 || bwait_cluster(bar(B1_RECVFREE + rs), ((st / 3) - 1) & 1, lim, fail));
                    if (!ok) {
                        if (!*fail) give_up();
                        break;
                    }
                    const uint32_t rbar = mapa(bar(B2_RECVFULL + rs), 1);
                    const uint32_t dst = mapa(sbase + K2_RECV + rs * RV_STAGE, 1);
                    const uint32_t src = sbase + K1_OUT + rs * OUT_BYTES;
                    mbar_arrive_expect_tx_remote_relaxed(rbar, 16384u);
                    bulk_copy_to_peer(dst + RV_W, src + OUT_W, 8192u, rbar);
                    bulk_copy_to_peer(dst + RV_TB, src + OUT_TB, 8192u, rbar);
                    KDA_TRACE_POINT(3, st);
                    shipped = st + 1;
                }
                // Copies still in flight read this CTA's memory: wait until the K2 CTA has
                // seen the last ones land (it relays each landing to OUTFREE).
                for (int st = (shipped >= 3 ? shipped - 3 : 0); st < shipped; ++st)
                    if (!mbar_wait_cluster(bar(B1_OUTFREE + st % 3), (st / 3) & 1, kDrainLimit))
                        record(p.status, kStatusTimeout);
            }
            __syncwarp();
        } else if (warp >= 4 && warp < 12) {
            // ---- elementwise warps (256 threads: channel pair x row quarter)
            const int et = tid - 128, pc = et & 63, qr = et >> 6;
            float4* scan = reinterpret_cast<float4*>(smem + K1_SCAN);
            for (int st = 0; st < nsteps; ++st) {
                const int s = st & 1;
                bool ok = !*fail;
                if (et == 0) {
                    ok = ok && bwait(bar(B1_IN_FULL + s), (st >> 1) & 1, lim, fail);
                    // Gram-A area s (read by W(st-2)) and the Gram-B rows written below
                    // (read by Gram(st-2) and Gram(st-3)) are free.
                    if (st >= 2)
                        ok = ok && bwait(bar(B1_WDONE + s), ((st >> 1) - 1) & 1, lim, fail) &&
                             bwait(bar(B1_GDONE + s), ((st >> 1) - 1) & 1, lim, fail);
                }
                if (named_bar_or(NB_E, 256, !ok)) {
                    if (et == 0 && !*fail) give_up();
                    break;
                }
                const unsigned char* in = smem + K1_IN + s * K1_IN_STAGE;
                const int C = step_rows(st);
                if (et == 0) KDA_TRACE_POINT(4, st);
                ETiles o;
                o.kt = smem + K1_A + s * K1_A_BYTES;
                o.kt_row0 = 0;
                o.qt = o.kt;
                o.qt_row0 = 32;
                o.kh = smem + K1_B + (st % 3) * K1_B_BYTES;
                o.kh_row0 = 0;
                o.kb = smem + K1_B + ((st + 1) % 3) * K1_B_BYTES;  // the next step's Kb_prev
                o.kb_row0 = 32;
                o.vt = nullptr;
                o.gc = nullptr;
                bool slow = e_step<4>(in + K1_IN_Q, in + K1_IN_K, nullptr,
                                      reinterpret_cast<const float*>(in + K1_IN_G), C, qr, pc, scan, NB_E, o,
                                      false);
                if (et < 32)  // beta of this step for the solve warps
                    reinterpret_cast<float*>(smem + K1_BETA)[s * 32 + et] =
                        reinterpret_cast<const float*>(in + K1_IN_BETA)[et];
                fence_proxy_async_smem();
                slow = named_bar_or(NB_E, 256, slow);
                if (et == 0) {
                    reinterpret_cast<volatile int32_t*>(smem + kSmSlow)[s] = slow ? 1 : 0;
                    KDA_TRACE_POINT(5, st);
                    mbar_arrive(bar(B1_EDONE + s));
                    // A slow step keeps its inputs until the exact Grams are formed.
                    if (!slow) mbar_arrive(bar(B1_IN_EMPTY + s));
                }
            }
        } else {
            // ---- TMEM warps 12..15 (lane quadrant = warp % 4).  Iteration `it` solves step it
            // (warps 12, 13) and then writes W of step it-1 (all four), whose MMA was issued
            // during the previous iteration, so no warp idles through an MMA round trip.
            const int quad = warp & 3;
            const uint32_t lanes = (uint32_t)(32 * quad) << 16;
            float* As = reinterpret_cast<float*>(smem + K1_AS);
            float* Xs = reinterpret_cast<float*>(smem + K1_XS);
            for (int it = 0; it <= nsteps; ++it) {
                bool ok = !*fail;
                const int st = it;
                if (quad < 2 && st < nsteps) {
                    const int s = st & 1;
                    unsigned char* out = smem + K1_OUT + (st % 3) * OUT_BYTES;
                    const float* beta = reinterpret_cast<const float*>(smem + K1_BETA) + s * 32;
                    // E(st) done (beta, slow flag), Gram(st) complete; out stage st % 3 free
                    // (its copy of step st-3 landed).
                    if (lane == 0) {
                        ok = ok && bwait(bar(B1_EDONE + s), (st >> 1) & 1, lim, fail) &&
                             bwait(bar(B1_GDONE + s), (st >> 1) & 1, lim, fail);
                        if (st >= 3) ok = ok && bwait_cluster(bar(B1_OUTFREE + st % 3), ((st / 3) - 1) & 1, lim, fail);
                    }
                    ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
                    ok = !named_bar_or(NB_SOLVE, 64, !ok);
                    if (!ok && tid == 32 * 12 && !*fail) give_up();
                    if (ok) {
                        if (tid == 32 * 12) KDA_TRACE_POINT(6, st);
                        tc_fence_after();
                        const bool slow = reinterpret_cast<volatile int32_t*>(smem + kSmSlow)[s] != 0;
                        const int r = lane;  // row of the step (Gram rows: Kt 0..31, Qt 32..63)
                        uint32_t a[32], x[32];
                        tmem_ld32(tmem + lanes + K1_TM_G + 64u * s, a);
                        tmem_ld32(tmem + lanes + K1_TM_G + 64u * s + 32, x);
                        tmem_wait_ld_regs<32>(a);
                        tmem_wait_ld_regs<32>(x);
                        if (tid == 32 * 12) KDA_TRACE_POINT(11, st);
                        if (quad == 0) {
                            const float br = beta[r];
                            if (!slow) {
#pragma unroll
                                for (int c = 0; c < 32; ++c) As[c * 32 + r] = c < r ? br * __uint_as_float(a[c]) : 0.f;
                            }
#pragma unroll
                            for (int c = 0; c < 32; ++c) Xs[c * 36 + r] = br * __uint_as_float(x[c]);
                        } else {
                            // Mq row r (lower incl. diagonal) and R row r, bf16 K-major
                            if (!slow) {
#pragma unroll
                                for (int g4 = 0; g4 < 4; ++g4) {
                                    uint32_t w[4];
#pragma unroll
                                    for (int u = 0; u < 4; ++u) {
                                        const int c = 8 * g4 + 2 * u;
                                        w[u] = pack_bf16(c <= r ? __uint_as_float(a[c]) : 0.f,
                                                         c + 1 <= r ? __uint_as_float(a[c + 1]) : 0.f);
                                    }
                                    *reinterpret_cast<uint4*>(out + OUT_MQ + km_off(r, 8 * g4)) =
                                        make_uint4(w[0], w[1], w[2], w[3]);
                                }
                            }
#pragma unroll
                            for (int g4 = 0; g4 < 4; ++g4) {
                                uint32_t w[4];
#pragma unroll
                                for (int u = 0; u < 4; ++u)
                                    w[u] = pack_bf16(__uint_as_float(x[8 * g4 + 2 * u]), __uint_as_float(x[8 * g4 + 2 * u + 1]));
                                *reinterpret_cast<uint4*>(out + OUT_PR + km_off(32 + r, 8 * g4)) =
                                    make_uint4(w[0], w[1], w[2], w[3]);
                            }
                        }
                        tc_fence_before();
                        named_bar_sync(NB_SOLVE, 64);
                        if (tid == 32 * 12) {
                            mbar_arrive(bar(B1_GREAD + s));
                            KDA_TRACE_POINT(12, st);
                        }
                        if (slow) {
                            // Exact Grams from the step's inputs, then release them.
                            k1_slow_grams(smem + K1_IN + s * K1_IN_STAGE, step_rows(st), tid - 32 * 12, As, beta,
                                          out + OUT_MQ);
                            named_bar_sync(NB_SOLVE, 64);
                            if (tid == 32 * 12) mbar_arrive(bar(B1_IN_EMPTY + s));
                        }
                        // Solves: warp 12 the columns of Tb, warp 13 those of P = T (beta o X).
                        float xs[32];
                        if (quad == 0) {
#pragma unroll
                            for (int i = 0; i < 32; ++i) xs[i] = i == lane ? 1.f : 0.f;
                        } else {
#pragma unroll
                            for (int i4 = 0; i4 < 8; ++i4) {
                                const float4 v = *reinterpret_cast<const float4*>(Xs + lane * 36 + 4 * i4);
                                xs[4 * i4] = v.x;
                                xs[4 * i4 + 1] = v.y;
                                xs[4 * i4 + 2] = v.z;
                                xs[4 * i4 + 3] = v.w;
                            }
                        }
                        solve32(As, xs);
                        if (tid == 32 * 12) KDA_TRACE_POINT(13, st);
                        if (tid == 32 * 13) KDA_TRACE_POINT(14, st);
                        if (quad == 0) {
                            const float bc = beta[lane];
#pragma unroll
                            for (int a4 = 0; a4 < 4; ++a4) {
                                uint32_t w[4];
#pragma unroll
                                for (int u = 0; u < 4; ++u)
                                    w[u] = pack_bf16(xs[8 * a4 + 2 * u] * bc, xs[8 * a4 + 2 * u + 1] * bc);
                                *reinterpret_cast<uint4*>(out + OUT_TB + tb_off(8 * a4, lane)) =
                                    make_uint4(w[0], w[1], w[2], w[3]);
                            }
                        } else {
#pragma unroll
                            for (int i = 0; i < 32; ++i)
                                *reinterpret_cast<__nv_bfloat16*>(out + OUT_PR + km_off(i, lane)) = __float2bfloat16_rn(xs[i]);
                        }
                        fence_proxy_async_smem();
                        named_bar_sync(NB_SOLVE, 64);
                        if (tid == 32 * 12) {
                            mbar_arrive(bar(B1_TBREADY + s));
                            KDA_TRACE_POINT(7, st);
                        }
                    }
                }
                // ---- all four: W^T of step it-1 from TMEM into its out stage (rows 0..31,
                // bf16).  Every TMEM warp reaches this barrier each iteration after the first,
                // so a failure seen by any of them ends the loop for all four together.
                const int ep = it - 1;
                if (ep < 0) continue;
                const int s = ep & 1;
                if (lane == 0 && ok) ok = !*fail && bwait(bar(B1_WDONE + s), (ep >> 1) & 1, lim, fail);
                ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
                if (named_bar_or(NB_EPI, 128, !ok)) {
                    if (tid == 32 * 12 && !*fail) give_up();
                    break;
                }
                tc_fence_after();
                {
                    unsigned char* out = smem + K1_OUT + (ep % 3) * OUT_BYTES;
                    uint32_t w[32];
                    tmem_ld32(tmem + lanes + K1_TM_W + 32u * s, w);
                    tmem_wait_ld_regs<32>(w);
                    const int ch = 32 * quad + lane;
#pragma unroll
                    for (int a4 = 0; a4 < 4; ++a4) {
                        uint32_t v[4];
#pragma unroll
                        for (int u = 0; u < 4; ++u)
                            v[u] = pack_bf16(__uint_as_float(w[8 * a4 + 2 * u]), __uint_as_float(w[8 * a4 + 2 * u + 1]));
                        *reinterpret_cast<uint4*>(out + OUT_W + tile_off(8 * a4, ch)) = make_uint4(v[0], v[1], v[2], v[3]);
                    }
                }
                fence_proxy_async_smem();
                tc_fence_before();
                named_bar_sync(NB_EPI, 128);
                if (tid == 32 * 12) {
                    mbar_arrive(bar(B1_OUTREADY + s));
                    KDA_TRACE_POINT(8, ep);
                }
            }
        }
    } else {
        // =============================================================== K2 CTA
        const uint32_t tS = tmem + K2_TM_S;
        auto tSA = [&](int i) { return tmem + K2_TM_SA + 64u * (uint32_t)i; };
        auto tACC = [&](int i) { return tmem + K2_TM_ACC + 64u * (uint32_t)i; };
        auto tDA = [&](int i) { return tmem + K2_TM_DA + 16u * (uint32_t)i; };
        auto recv = [&](int st) { return sbase + K2_RECV + (uint32_t)(st % 3) * RV_STAGE; };
        auto stage_ready = [&](int st) {  // K1's part landed and the local part written
            return bwait(bar(B2_RECVFULL + st % 3), (st / 3) & 1, lim, fail) &&
                   bwait(bar(B2_LOCALREADY + st % 3), (st / 3) & 1, lim, fail);
        };
        if (warp == 0) {
            // ---- TMA producer: q, k, v, g of each step.
            int issued = 0;
            if (lane == 0) {
                for (int st = 0; st < nsteps; ++st) {
                    const int s = st & 1;
                    if (st >= 2 && !bwait(bar(B2_IN_EMPTY + s), ((st >> 1) - 1) & 1, lim, fail)) {
                        if (!*fail) give_up();
                        break;
                    }
                    const uint32_t dst = sbase + K2_IN + s * K2_IN_STAGE;
                    const int32_t t0 = (int32_t)(bos + (int64_t)st * kBlk);
                    mbar_arrive_expect_tx(bar(B2_IN_FULL + s), 40960u);
                    tma_load_3d(dst + K2_IN_Q, &tm_q, bar(B2_IN_FULL + s), 0, hq, t0);
                    tma_load_3d(dst + K2_IN_K, &tm_k, bar(B2_IN_FULL + s), 0, hk, t0);
                    tma_load_3d(dst + K2_IN_V, &tm_v, bar(B2_IN_FULL + s), 0, h, t0);
                    tma_load_3d(dst + K2_IN_G, &tm_g, bar(B2_IN_FULL + s), 0, h, t0);
                    KDA_TRACE_POINT(16, st);
                    issued = st + 1;
                }
                for (int st = (issued >= 2 ? issued - 2 : 0); st < issued; ++st)
                    if (!mbar_wait(bar(B2_IN_FULL + (st & 1)), (st >> 1) & 1, kDrainLimit))
                        record(p.status, kStatusTimeout);
            }
            __syncwarp();
        } else if (warp == 3) {
            // ---- relay: each landed step frees K1's out stage it came from.
            if (lane == 0) {
                for (int st = 0; st < nsteps; ++st) {
                    // Keep relaying after a failure elsewhere (K1 waits for its copies), but
                    // with the drain bound once this CTA has failed.
                    const bool ok = mbar_wait(bar(B2_RECVFULL + st % 3), (st / 3) & 1, *fail ? 4096 : lim);
                    if (!ok) {
                        if (!*fail) give_up();
                        break;
                    }
                    mbar_arrive_remote_relaxed(mapa(bar(B1_OUTFREE + st % 3), 0));
                    KDA_TRACE_POINT(17, st);
                }
            }
            __syncwarp();
        } else if (warp >= 12) {
            // ---- Qt, Kb, V operand and e^{gam_C} of each step (128 threads: channel pair x row half)
            const int et = tid - 384, pc = et & 63, hf = et >> 6;
            float4* scan = reinterpret_cast<float4*>(smem + K2_SCAN);
            for (int st = 0; st < nsteps; ++st) {
                const int s = st & 1;
                bool ok = !*fail;
                if (et == 0) {
                    ok = ok && bwait(bar(B2_IN_FULL + s), (st >> 1) & 1, lim, fail);
                    if (st >= 3) ok = ok && bwait(bar(B2_LOCALFREE + st % 3), ((st / 3) - 1) & 1, lim, fail);
                }
                if (named_bar_or(NB_ELITE, 128, !ok)) {
                    if (et == 0 && !*fail) give_up();
                    break;
                }
                const unsigned char* in = smem + K2_IN + s * K2_IN_STAGE;
                unsigned char* rv = smem + K2_RECV + (st % 3) * RV_STAGE;
                if (et == 0) KDA_TRACE_POINT(18, st);
                ETiles o;
                o.kt = nullptr;
                o.kt_row0 = 0;
                o.qt = rv + RV_W;  // Qt is rows 32..63 of the MMA1 operand [W ; Qt]
                o.qt_row0 = 32;
                o.kb = rv + RV_KB;
                o.kb_row0 = 0;
                o.kh = nullptr;
                o.kh_row0 = 0;
                o.vt = rv + RV_V;
                o.gc = reinterpret_cast<float*>(rv + RV_GC);
                e_step<2>(in + K2_IN_Q, in + K2_IN_K, in + K2_IN_V, reinterpret_cast<const float*>(in + K2_IN_G),
                          step_rows(st), hf, pc, scan, NB_ELITE, o, zero_v);
                fence_proxy_async_smem();
                named_bar_sync(NB_ELITE, 128);
                if (et == 0) {
                    mbar_arrive(bar(B2_LOCALREADY + st % 3));
                    KDA_TRACE_POINT(19, st);
                    mbar_arrive(bar(B2_IN_EMPTY + s));
                }
            }
        } else if (warp == 1 || warp == 2) {
            // ---- MMA1 issuers: ACC(st) += D_st^T [W ; Qt]^T over all 128 keys; warp 1 the W
            // rows (columns 0..31, on the chain), warp 2 the Qt rows (columns 32..63).  Each
            // accumulator column has one issuer adding in a fixed order, so results are
            // bit-reproducible.
            const int nh = warp - 1;
            const uint32_t id1 = idesc_bf16(128, 32) | kIdescBMn;
            for (int st = 0; st < nsteps; ++st) {
                bool ok = true;
                if (lane == 0)
                    ok = bwait(bar(B2_SAREADY + (st & 1)), (st >> 1) & 1, lim, fail) &&
                         bwait(bar(B2_LOOK), st & 1, lim, fail) && stage_ready(st);
                if (__any_sync(0xffffffffu, !ok)) {
                    if (lane == 0 && !*fail) give_up();
                    break;
                }
                tc_fence_after();
                if (elect_one()) {
                    const uint32_t b1 = recv(st) + RV_W + (uint32_t)nh * 4u * kRG;  // rows 0..31 or 32..63
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk)
                        mma_ts(tACC(st % 3) + 32u * nh, tSA(st & 1) + 8u * kk, sdesc(b1 + kk * 256, 128, kRG), id1, 1);
                    tc_commit(bar(B2_MMA1));
                    if (nh == 0) KDA_TRACE_POINT(20, st);
                }
                __syncwarp();
            }
            if (elect_one()) tc_commit(bar(B2_DRAIN));
            __syncwarp();
            if (!mbar_wait(bar(B2_DRAIN), 0, kDrainLimit) && lane == 0) record(p.status, kStatusTimeout);
        } else if (warp >= 4 && warp < 8) {
            // ---- delta warps (thread = value column j)
            const int quad = warp & 3, j = 32 * quad + lane;
            const uint32_t lanes = (uint32_t)(32 * quad) << 16;
            const bool leader = warp == 4 && lane == 0;
            const uint32_t idU = idesc_bf16(128, 32) | kIdescBMn | kIdescNegB;
            const uint32_t id32 = idesc_bf16(128, 32);
            // U(st) and the lookahead terms of step st into ACC(st) (lookahead operands are
            // delta_{st-1} in DA((st-1)&1) and [P ; R] of step st).
            auto issue_look = [&](int st) {
                const uint32_t rv = recv(st);
                const uint32_t acc = tACC(st % 3), da = tDA((st + 1) & 1);
#pragma unroll
                for (int kk = 0; kk < 2; ++kk)  // ACC_W = -Vt Tb^T   (U)
                    mma_ss(acc, sdesc(rv + RV_V + kk * 2 * kRG, kRG, 128), sdesc(rv + RV_TB + kk * 256, 128, 512),
                           idU, kk > 0);
#pragma unroll
                for (int kk = 0; kk < 2; ++kk)  // ACC_W += delta^T P^T
                    mma_ts(acc, da + 8u * kk, sdesc(rv + RV_PR + kk * 256, 128, 512), id32, 1);
#pragma unroll
                for (int kk = 0; kk < 2; ++kk)  // ACC_Q = delta^T R^T
                    mma_ts(acc + 32, da + 8u * kk, sdesc(rv + RV_PR + 2048 + kk * 256, 128, 512), id32, kk > 0);
                tc_commit(bar(B2_L));
            };
            // Output rows of step st: ACC_Q * scale -> bf16, through a tile stored by TMA
            // (full steps) or plain stores (a ragged last step).
            auto emit_out = [&](int st) {
                uint32_t o[32];
                tmem_ld32(tACC(st % 3) + lanes + 32, o);
                tmem_wait_ld_regs<32>(o);
                const int C = step_rows(st);
                const int64_t t0 = bos + (int64_t)st * kBlk;
                if (C == kBlk) {
                    __nv_bfloat16* tile = reinterpret_cast<__nv_bfloat16*>(smem + K2_OTILE + (st & 1) * 8192);
#pragma unroll
                    for (int r = 0; r < 32; ++r) tile[r * 128 + j] = __float2bfloat16_rn(p.scale * __uint_as_float(o[r]));
                    fence_proxy_async_smem();
                    named_bar_sync(NB_DELTA, 128);
                    if (leader) {
                        tma_store_3d(&tm_out, sbase + K2_OTILE + (st & 1) * 8192, 0, ho, (int32_t)t0);
                        bulk_commit();
                        bulk_wait_read<1>();  // the other tile's store has read its source
                    }
                } else {
#pragma unroll
                    for (int r = 0; r < 32; ++r)
                        if (r < C)
                            p.out[((t0 + r) * Ho + ho) * kD + j] = __float2bfloat16_rn(p.scale * __uint_as_float(o[r]));
                }
            };
            bool ok = true, alive = true;
            if (nsteps > 0) {
                // delta_{-1} = 0
                uint32_t z[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) z[i] = 0u;
                tmem_st16(tDA(1) + lanes, z);
                tmem_wait_st();
                tc_fence_before();
                named_bar_sync(NB_DELTA, 128);
                if (leader) {
                    ok = stage_ready(0);
                    if (ok) {
                        tc_fence_after();
                        issue_look(0);
                        mbar_arrive(bar(B2_LOOK));
                    } else if (!*fail) {
                        give_up();
                    }
                }
            }
            for (int st = 0; st < nsteps; ++st) {
                if (lane == 0)
                    ok = !*fail && bwait(bar(B2_L), st & 1, lim, fail) && bwait(bar(B2_MMA1), st & 1, lim, fail);
                ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
                if (named_bar_or(NB_DELTA, 128, !ok)) {
                    if (leader && !*fail) give_up();
                    alive = false;
                    break;
                }
                tc_fence_after();
                {
                    uint32_t a[32], d[16];                if (leader) KDA_TRACE_POINT(21, st);

                    tmem_ld32(tACC(st % 3) + lanes, a);
                    tmem_wait_ld_regs<32>(a);
#pragma unroll
                    for (int i = 0; i < 16; ++i)
                        d[i] = pack_bf16(-__uint_as_float(a[2 * i]), -__uint_as_float(a[2 * i + 1]));
                    tmem_st16(tDA(st & 1) + lanes, d);
                    tmem_wait_st();
                }
                tc_fence_before();
                named_bar_sync(NB_DELTA, 128);
                if (leader) {
                    mbar_arrive(bar(B2_DELTA));  // the decay warps issue the state update
                    KDA_TRACE_POINT(22, st);
                    if (st + 1 < nsteps) {
                        if (stage_ready(st + 1)) {
                            tc_fence_after();
                            issue_look(st + 1);
                            mbar_arrive(bar(B2_LOOK));
                            KDA_TRACE_POINT(23, st);
                        } else if (!*fail) {
                            give_up();
                        }
                    }
                }
                // Output of the previous step (its Mq term completed with SDONE(st-1)).
                if (st > 0 && with_out) {
                    bool okp = true;
                    if (lane == 0) okp = bwait(bar(B2_SDONE + ((st - 1) & 1)), ((st - 1) >> 1) & 1, lim, fail);
                    okp = __shfl_sync(0xffffffffu, okp ? 1 : 0, 0) != 0;
                    if (named_bar_or(NB_DELTA, 128, !okp)) {
                        if (leader && !*fail) give_up();
                        alive = false;
                        break;
                    }
                    tc_fence_after();
                    emit_out(st - 1);
                }
            }
            if (nsteps > 0 && with_out && alive) {
                bool okp = true;
                if (lane == 0) okp = bwait(bar(B2_SDONE + ((nsteps - 1) & 1)), ((nsteps - 1) >> 1) & 1, lim, fail);
                okp = __shfl_sync(0xffffffffu, okp ? 1 : 0, 0) != 0;
                if (!named_bar_or(NB_DELTA, 128, !okp)) {
                    tc_fence_after();
                    emit_out(nsteps - 1);
                } else if (leader && !*fail) {
                    give_up();
                }
            }
            if (leader) bulk_wait0();  // output stores complete before exit
            tmem_wait_ld();
            if (warp == 4) {
                if (elect_one()) tc_commit(bar(B2_DRAIN));
                __syncwarp();
                if (!mbar_wait(bar(B2_DRAIN), 0, kDrainLimit) && lane == 0) record(p.status, kStatusTimeout);
            }
        } else {
            // ---- decay warps 8..11 (thread = value column j): the state S^T in TMEM (lane j,
            // column i = key), its in-place decay, its bf16 copy and the state update.
            const int quad = warp & 3, j = 32 * quad + lane;
            const uint32_t lanes = (uint32_t)(32 * quad) << 16;
            const bool leader = warp == 8 && lane == 0;
            const uint32_t id128 = idesc_bf16(128, 128), id32 = idesc_bf16(128, 32);
            const size_t soff = ((size_t)row * p.H + h) * kD * kD;
            size_t foff = soff;
            bool write_final = p.sfin != nullptr && state_owner;
            if (p.flags & kFlagFinalLastSeg) {
                write_final = write_final && seg_id == seg_count - 1;
                foff = ((size_t)seq_id * p.H + h) * kD * kD;
            }
            auto s0_at = [&](int i) -> float {
                if (p.flags & kFlagIdentityS0) return i == j ? 1.f : 0.f;
                if (p.s0 == nullptr) return 0.f;
                const size_t idx = soff + (size_t)i * kD + j;
                return p.s0_bf16 ? __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(p.s0)[idx]) : p.s0[idx];
            };
            auto store_final = [&](int i, float v) {
                const size_t idx = foff + (size_t)i * kD + j;
                if (p.sfin_bf16) reinterpret_cast<__nv_bfloat16*>(p.sfin)[idx] = __float2bfloat16_rn(v);
                else p.sfin[idx] = v;
            };
            if (nsteps == 0) {
                // No tokens: the final state is the initial state.
                if (write_final)
                    for (int i = 0; i < kD; ++i) store_final(i, s0_at(i));
            } else {
                // Initial state S0[i][j] -> S^T (lane j, column i) and its bf16 copy SA(0).
#pragma unroll 1
                for (int pass = 0; pass < 4; ++pass) {
                    uint32_t v[32], pk[16];
#pragma unroll
                    for (int i = 0; i < 32; ++i) v[i] = __float_as_uint(s0_at(32 * pass + i));
#pragma unroll
                    for (int i = 0; i < 16; ++i) pk[i] = pack_bf16(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1]));
                    tmem_st32(tS + lanes + 32u * pass, v);
                    tmem_st16(tSA(0) + lanes + 16u * pass, pk);
                }
                tmem_wait_st();
                tc_fence_before();
                named_bar_sync(NB_DECAY, 128);
                if (leader) mbar_arrive(bar(B2_SAREADY + 0));
                if ((p.debug_flags & 1) && warp == 8 && !mbar_wait(bar(B2_NEVER), 0, lim) && lane == 0) give_up();
            }
            bool ok = true, alive = true;
            for (int st = 0; st < nsteps; ++st) {
                const int rs = st % 3;
                if (lane == 0) {
                    ok = !*fail;
                    if (st > 0) ok = ok && bwait(bar(B2_SDONE + ((st - 1) & 1)), ((st - 1) >> 1) & 1, lim, fail);
                    ok = ok && bwait(bar(B2_LOCALREADY + rs), (st / 3) & 1, lim, fail);
                }
                ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
                if (named_bar_or(NB_DECAY, 128, !ok)) {
                    if (leader && !*fail) give_up();
                    alive = false;
                    break;
                }
                if (leader) KDA_TRACE_POINT(24, st);
                if (leader && st > 0) {
                    // Step st-1 is consumed: K1 may ship step st+2 into its stage, and the
                    // local part of that stage may be rewritten.
                    mbar_arrive_remote_relaxed(mapa(bar(B1_RECVFREE + (st - 1) % 3), 0));
                    mbar_arrive(bar(B2_LOCALFREE + (st - 1) % 3));
                }
                tc_fence_after();
                // D_{st+1} = Diag(e^{gam_C(st)}) S_st in place, and its bf16 copy for MMA1(st+1).
                const float4* gc4 = reinterpret_cast<const float4*>(smem + K2_RECV + rs * RV_STAGE + RV_GC);
                const bool next = st + 1 < nsteps;
#pragma unroll 1
                for (int pass = 0; pass < 4; ++pass) {
                    uint32_t v[32], pk[16];
                    tmem_ld32(tS + lanes + 32u * pass, v);
                    tmem_wait_ld_regs<32>(v);
#pragma unroll
                    for (int i4 = 0; i4 < 8; ++i4) {
                        const float4 gv = gc4[8 * pass + i4];
                        float a0 = __uint_as_float(v[4 * i4]), a1 = __uint_as_float(v[4 * i4 + 1]);
                        float a2 = __uint_as_float(v[4 * i4 + 2]), a3 = __uint_as_float(v[4 * i4 + 3]);
                        mul2(a0, a1, gv.x, gv.y);
                        mul2(a2, a3, gv.z, gv.w);
                        v[4 * i4] = __float_as_uint(a0);
                        v[4 * i4 + 1] = __float_as_uint(a1);
                        v[4 * i4 + 2] = __float_as_uint(a2);
                        v[4 * i4 + 3] = __float_as_uint(a3);
                    }
                    tmem_st32(tS + lanes + 32u * pass, v);
                    if (next) {
#pragma unroll
                        for (int i = 0; i < 16; ++i) pk[i] = pack_bf16(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1]));
                        tmem_st16(tSA((st + 1) & 1) + lanes + 16u * pass, pk);
                    }
                }
                tmem_wait_st();
                tc_fence_before();
                named_bar_sync(NB_DECAY, 128);
                if (leader) {
                    // S += Kb^T delta_st (onto D_{st+1}) and ACC_Q(st) += delta^T Mq^T.
                    KDA_TRACE_POINT(25, st);
                    bool okd = bwait(bar(B2_DELTA), st & 1, lim, fail);
                    if (okd) {
                        tc_fence_after();
                        const uint32_t rv = recv(st), da = tDA(st & 1);
#pragma unroll
                        for (int kk = 0; kk < 2; ++kk)
                            mma_ts(tS, da + 8u * kk, sdesc(rv + RV_KB + kk * 2 * kRG, kRG, 128), id128, 1);
                        if (with_out) {
#pragma unroll
                            for (int kk = 0; kk < 2; ++kk)
                                mma_ts(tACC(rs) + 32, da + 8u * kk, sdesc(rv + RV_MQ + kk * 256, 128, 512), id32, 1);
                        }
                        tc_commit(bar(B2_SDONE + (st & 1)));
                        KDA_TRACE_POINT(26, st);
                        if (next) mbar_arrive(bar(B2_SAREADY + ((st + 1) & 1)));
                    } else if (!*fail) {
                        give_up();
                    }
                }
            }
            if (nsteps > 0 && alive) {
                bool okf = true;
                if (lane == 0) okf = bwait(bar(B2_SDONE + ((nsteps - 1) & 1)), ((nsteps - 1) >> 1) & 1, lim, fail);
                okf = __shfl_sync(0xffffffffu, okf ? 1 : 0, 0) != 0;
                if (!named_bar_or(NB_DECAY, 128, !okf)) {
                    tc_fence_after();
                    if (write_final) {
#pragma unroll 1
                        for (int pass = 0; pass < 4; ++pass) {
                            uint32_t v[32];
                            tmem_ld32(tS + lanes + 32u * pass, v);
                            tmem_wait_ld_regs<32>(v);
#pragma unroll
                            for (int i = 0; i < 32; ++i) store_final(32 * pass + i, __uint_as_float(v[i]));
                        }
                    }
                } else if (leader && !*fail) {
                    give_up();
                }
            }
            tmem_wait_ld();
            tmem_wait_st();
            if (warp == 8) {
                if (elect_one()) tc_commit(bar(B2_DRAIN));
                __syncwarp();
                if (!mbar_wait(bar(B2_DRAIN), 0, kDrainLimit) && lane == 0) record(p.status, kStatusTimeout);
            }
        }
    }

    tc_fence_before();
    cluster_sync();  // neither CTA leaves while its peer may still access its memory
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, rank == 0 ? K1_TM_COLS : K2_TM_COLS);
    }
}

}  // namespace

size_t serial_smem_bytes() { return kSmemBytes; }
int serial_block_threads() { return kThreads; }
const void* serial_kernel_symbol() { return reinterpret_cast<const void*>(&kda_fwd_kernel<false>); }
const void* grouped_kernel_symbol() { return reinterpret_cast<const void*>(&kda_fwd_kernel<true>); }

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
        return cudaLaunchKernelEx(&cfg, kda_fwd_kernel<true>, maps.q, maps.k, maps.v, maps.g, maps.out, p);
    return cudaLaunchKernelEx(&cfg, kda_fwd_kernel<false>, maps.q, maps.k, maps.v, maps.g, maps.out, p);
}

}  // namespace kda
