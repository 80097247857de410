// kda_fwd_tc.cu -- fused K1 + K2 KDA forward prefill for sm_103a: TMA-staged chunk
// tiles, tcgen05 MMAs with the state held in tensor memory (TMEM) across all chunks.
//
// The method (cuLA PR #103 "feat(kda/sm90): FlashKDA prefill port + intracard-CP
// prefill", commit notes: "K1 prepares decayed q/k, beta and the WY inverse; K2 runs
// the inter-chunk recurrence. CHUNK=16, D=128, forward only").  For a chunk of C <= 16
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
// exp(gam_r - gam_ref) exp(gam_ref - gam_s); each factor stays in fp32 range while
// the log-decay accumulated over 8 consecutive tokens of a channel is above ~-80.
//
// Mapping (transposed so the 128-wide value dim is the MMA's M):
//   TMEM holds S^T (lane j = value column, column i = key row) in fp32.
//   MMA1: D1[j][0:32]  = S^T[j][:] . [W ; Qtil]^T   (A = bf16 copy of S^T in TMEM,
//                                                    B = [W ; Qtil] in shared memory)
//   delta^T = U^T - D1[:, 0:16]   (epilogue threads, written back to TMEM as bf16)
//   MMA2: S^T += delta^T . Kbar   (after the epilogue scaled S^T by exp(gam_C))
//   MMA3: D1[:, 16:32] += delta^T . Mq^T;  O^T = scale * D1[:, 16:32]
// Warp roles (448 threads): warp 0 TMA producer; warp 1 MMA issuer and TMEM owner;
// warps 2-5 K1 (cumulative decay, decayed operands, in-chunk Grams and the WY
// solve; the 16x16 products use mma.sync because tcgen05's smallest M is 64);
// warps 6-13 the K2 epilogue (state conversion/decay, delta, output).
// Every wait is bounded: on exhaustion the kernel records KDA_ERR_DEVICE_TIMEOUT
// in the status word, drains its in-flight copies and MMAs and exits.
#include <cuda.h>

#include "kda_internal.cuh"
#include "kda_ptx.cuh"

namespace kda {
namespace {

using namespace ptx;

constexpr int kThreads = 448;
constexpr int kRef = 7;
constexpr uint32_t kTmemCols = 512;
// Bound of the waits that drain in-flight copies and MMAs before exit; independent of
// the caller's wait limit so that an early exit never leaves asynchronous work behind.
constexpr int64_t kDrainLimit = 1ll << 24;

// TMEM column map
constexpr uint32_t kColS = 0;     // S^T fp32, 128 columns
constexpr uint32_t kColSA = 128;  // S^T bf16 pairs, 64 columns (MMA1 A operand)
constexpr uint32_t kColD1 = 192;  // two 32-column buffers (MMA1/MMA3 accumulators)
constexpr uint32_t kColDA = 256;  // delta^T bf16 pairs, 8 columns (MMA2/MMA3 A operand)

// Shared memory map (bytes)
constexpr int kInQ = 0, kInK = 4096, kInV = 8192, kInG = 12288, kInBytes = 20480;
constexpr uint32_t kTxBytes = kInBytes;
constexpr int kB1 = 0, kB2 = 8192, kB3 = 12288, kU = 12800, kGC = 20992, kOutBytes = 21504;
constexpr uint32_t kLbo = 128, kSboB1 = 2048, kSboB2 = 256, kSboB3 = 256;
constexpr int kStRow = 272, kStArr = 16 * kStRow;  // padded bf16 staging rows (136 elems)
enum { ST_KQ = 0, ST_QQ, ST_KK, ST_KT, ST_VV, ST_QT, ST_NUM };
constexpr int kSmIn = 0;                               // 2 input stages
constexpr int kSmOut = kSmIn + 2 * kInBytes;           // 2 K1 output stages
constexpr int kSmSt = kSmOut + 2 * kOutBytes;          // staging
constexpr int kSmA = kSmSt + ST_NUM * kStArr;          // fp32 16x16
constexpr int kSmTb = kSmA + 1024;                     // bf16 16x24
constexpr int kSmBeta = kSmTb + 768;                   // fp32 16
constexpr int kSmBar = kSmBeta + 64;                   // mbarriers
constexpr int kNumBars = 16;
constexpr int kSmTmemSlot = kSmBar + kNumBars * 8;
constexpr int kSmemBytes = kSmTmemSlot + 16;
enum {
    BAR_IN_FULL = 0, BAR_IN_EMPTY = 2, BAR_K1_FULL = 4, BAR_K1_EMPTY = 6,
    BAR_SA = 8, BAR_D1 = 9, BAR_DL = 10, BAR_SDONE = 11, BAR_DRAIN = 12
};
constexpr uint32_t kNamedK1 = 1;

__device__ __forceinline__ uint32_t b1_off(int n, int k) {
    return (n >> 3) * kSboB1 + (k >> 3) * kLbo + (n & 7) * 16 + (k & 7) * 2;
}
__device__ __forceinline__ uint32_t b3_off(int n, int k) {
    return (n >> 3) * kSboB3 + (k >> 3) * kLbo + (n & 7) * 16 + (k & 7) * 2;
}

__device__ __forceinline__ void record(int32_t* status, int32_t code) {
    atomicCAS(status, kStatusOk, code);
}

__device__ __forceinline__ float bf_lo(uint32_t x) { return __uint_as_float(x << 16); }
__device__ __forceinline__ float bf_hi(uint32_t x) { return __uint_as_float(x & 0xffff0000u); }

__global__ void __launch_bounds__(kThreads, 1)
kda_fwd_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_g,
                  const FwdParams p) {
    extern __shared__ __align__(1024) unsigned char smem[];
    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int h = blockIdx.x % p.H;
    const int n = blockIdx.x / p.H;
    int64_t bos, eos;
    if (!seq_range(p, n, bos, eos)) return;
    const int64_t H = p.H;
    const int nchunks = (int)((eos - bos + kChunk - 1) / kChunk);
    const int64_t lim = p.wait_limit;
    const uint32_t sbase = smem_u32(smem);
    const uint32_t bars = sbase + kSmBar;
    auto bar = [&](int i) { return bars + 8u * (uint32_t)i; };
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kSmTmemSlot);

    if (tid == 0) {
        for (int s = 0; s < 2; ++s) {
            mbar_init(bar(BAR_IN_FULL + s), 1);
            mbar_init(bar(BAR_IN_EMPTY + s), 1);
            mbar_init(bar(BAR_K1_FULL + s), 128);
            mbar_init(bar(BAR_K1_EMPTY + s), 256);
        }
        mbar_init(bar(BAR_SA), 256);
        mbar_init(bar(BAR_D1), 1);
        mbar_init(bar(BAR_DL), 256);
        mbar_init(bar(BAR_SDONE), 1);
        mbar_init(bar(BAR_DRAIN), 1);
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), kTmemCols);
        tmem_relinquish();
    }
    if (warp == 0 && lane == 0 && nchunks > 0) {
        prefetch_tmap(&tm_q);
        prefetch_tmap(&tm_k);
        prefetch_tmap(&tm_v);
        prefetch_tmap(&tm_g);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            int issued = 0;
            for (int c = 0; c < nchunks; ++c) {
                const int s = c & 1;
                if (c >= 2 && !mbar_wait(bar(BAR_IN_EMPTY + s), ((c >> 1) - 1) & 1, lim)) {
                    record(p.status, kStatusTimeout);
                    break;
                }
                const uint32_t dst = sbase + kSmIn + s * kInBytes;
                const int32_t t0 = (int32_t)(bos + (int64_t)c * kChunk);
                mbar_arrive_expect_tx(bar(BAR_IN_FULL + s), kTxBytes);
                tma_load_3d(dst + kInQ, &tm_q, bar(BAR_IN_FULL + s), 0, h, t0);
                tma_load_3d(dst + kInK, &tm_k, bar(BAR_IN_FULL + s), 0, h, t0);
                tma_load_3d(dst + kInV, &tm_v, bar(BAR_IN_FULL + s), 0, h, t0);
                tma_load_3d(dst + kInG, &tm_g, bar(BAR_IN_FULL + s), 0, h, t0);
                issued = c + 1;
            }
            // Drain: every issued load must have landed before the CTA exits.
            for (int c = (issued >= 2 ? issued - 2 : 0); c < issued; ++c)
                if (!mbar_wait(bar(BAR_IN_FULL + (c & 1)), (c >> 1) & 1, kDrainLimit))
                    record(p.status, kStatusTimeout);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            const uint32_t idesc1 = idesc_bf16(128, 32);
            const uint32_t idesc2 = idesc_bf16(128, 128);
            const uint32_t idesc3 = idesc_bf16(128, 16);
            for (int c = 0; c < nchunks; ++c) {
                const int ks = c & 1;
                const uint32_t ob = sbase + kSmOut + ks * kOutBytes;
                if (!mbar_wait(bar(BAR_K1_FULL + ks), (c >> 1) & 1, lim) ||
                    !mbar_wait(bar(BAR_SA), c & 1, lim)) {
                    record(p.status, kStatusTimeout);
                    break;
                }
                tc_fence_after();
                const uint32_t d1 = tmem + kColD1 + 32u * (uint32_t)(c & 1);
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)
                    mma_ts(d1, tmem + kColSA + 8u * kk, sdesc(ob + kB1 + kk * 2 * kLbo, kLbo, kSboB1),
                           idesc1, kk > 0);
                tc_commit(bar(BAR_D1));
                if (!mbar_wait(bar(BAR_DL), c & 1, lim)) {
                    record(p.status, kStatusTimeout);
                    break;
                }
                tc_fence_after();
                mma_ts(tmem + kColS, tmem + kColDA, sdesc(ob + kB2, kLbo, kSboB2), idesc2, 1);
                mma_ts(d1 + 16, tmem + kColDA, sdesc(ob + kB3, kLbo, kSboB3), idesc3, 1);
                tc_commit(bar(BAR_SDONE));
            }
            // Drain every MMA issued before TMEM is released.
            tc_commit(bar(BAR_DRAIN));
            if (!mbar_wait(bar(BAR_DRAIN), 0, kDrainLimit)) record(p.status, kStatusTimeout);
        }
    } else if (warp < 6) {
        // ------------------------------------------------------------ K1 (128 threads)
        const int kt = tid - 64;          // 0..127
        const int kw = kt >> 5;           // K1 warp 0..3
        const int pc = kt & 63;           // channel pair: channels 2pc, 2pc+1
        const int hr = kt >> 6;           // row half: rows 8hr .. 8hr+7
        unsigned char* st = smem + kSmSt;
        float* Asm = reinterpret_cast<float*>(smem + kSmA);
        __nv_bfloat16* Tb = reinterpret_cast<__nv_bfloat16*>(smem + kSmTb);
        float* bet = reinterpret_cast<float*>(smem + kSmBeta);
        for (int c = 0; c < nchunks; ++c) {
            const int s = c & 1, ks = c & 1;
            bool ok = mbar_wait(bar(BAR_IN_FULL + s), (c >> 1) & 1, lim);
            if (ok && c >= 2) ok = mbar_wait(bar(BAR_K1_EMPTY + ks), ((c >> 1) - 1) & 1, lim);
            if (named_bar_or(kNamedK1, 128, !ok)) {
                if (kt == 0) record(p.status, kStatusTimeout);
                break;
            }
            const int64_t t0 = bos + (int64_t)c * kChunk;
            const int C = (eos - t0 < kChunk) ? (int)(eos - t0) : kChunk;
            const unsigned char* in = smem + kSmIn + s * kInBytes;
            unsigned char* ob = smem + kSmOut + ks * kOutBytes;
            if (kt < kChunk) bet[kt] = kt < C ? __bfloat162float(p.beta[(t0 + kt) * H + h]) : 0.f;

            // Phase 1: cumulative decay and decayed operands for channels 2pc, 2pc+1.
            const float2* g2 = reinterpret_cast<const float2*>(in + kInG);
            float ga[kChunk], gb[kChunk];
            {
                float a0 = 0.f, a1 = 0.f;
#pragma unroll
                for (int r = 0; r < kChunk; ++r) {
                    const float2 gv = r < C ? g2[r * 64 + pc] : make_float2(0.f, 0.f);
                    a0 += gv.x;
                    a1 += gv.y;
                    ga[r] = a0;
                    gb[r] = a1;
                }
            }
            const float ref0 = ga[kRef], ref1 = gb[kRef];
            float gh0[8], gh1[8];  // this thread's rows, selected with constant indices
#pragma unroll
            for (int rr = 0; rr < 8; ++rr) {
                gh0[rr] = hr ? ga[8 + rr] : ga[rr];
                gh1[rr] = hr ? gb[8 + rr] : gb[rr];
            }
            const float eref0 = __expf(ref0), eref1 = __expf(ref1);
            const float ecr0 = __expf(ga[kChunk - 1] - ref0), ecr1 = __expf(gb[kChunk - 1] - ref1);
            if (hr == 0) {
                float* gc = reinterpret_cast<float*>(ob + kGC);
                gc[2 * pc] = __expf(ga[kChunk - 1]);
                gc[2 * pc + 1] = __expf(gb[kChunk - 1]);
            }
            const uint32_t* q2 = reinterpret_cast<const uint32_t*>(in + kInQ);
            const uint32_t* k2 = reinterpret_cast<const uint32_t*>(in + kInK);
            const uint32_t* v2 = reinterpret_cast<const uint32_t*>(in + kInV);
            uint32_t kb0[4], kb1[4];
#pragma unroll
            for (int rr = 0; rr < 8; ++rr) {
                const int r = 8 * hr + rr;
                const bool valid = r < C;
                const uint32_t qv = valid ? q2[r * 64 + pc] : 0u;
                const uint32_t kv = valid ? k2[r * 64 + pc] : 0u;
                const uint32_t vv = valid ? v2[r * 64 + pc] : 0u;
                const float k0 = bf_lo(kv), k1 = bf_hi(kv), q0 = bf_lo(qv), q1 = bf_hi(qv);
                const float up0 = __expf(gh0[rr] - ref0), up1 = __expf(gh1[rr] - ref1);
                const float dn0 = __expf(ref0 - gh0[rr]), dn1 = __expf(ref1 - gh1[rr]);
                uint32_t* row = reinterpret_cast<uint32_t*>(st + r * kStRow) + pc;
                row[ST_KQ * kStArr / 4] = pack_bf16(k0 * up0, k1 * up1);
                row[ST_QQ * kStArr / 4] = pack_bf16(q0 * up0, q1 * up1);
                row[ST_KK * kStArr / 4] = pack_bf16(k0 * dn0, k1 * dn1);
                row[ST_KT * kStArr / 4] = pack_bf16(k0 * up0 * eref0, k1 * up1 * eref1);
                row[ST_QT * kStArr / 4] = pack_bf16(q0 * up0 * eref0, q1 * up1 * eref1);
                row[ST_VV * kStArr / 4] = vv;
                const float kbar0 = k0 * dn0 * ecr0, kbar1 = k1 * dn1 * ecr1;
                if (rr & 1) {
                    kb0[rr >> 1] |= pack_bf16(0.f, kbar0) & 0xffff0000u;
                    kb1[rr >> 1] |= pack_bf16(0.f, kbar1) & 0xffff0000u;
                } else {
                    kb0[rr >> 1] = pack_bf16(kbar0, 0.f) & 0xffffu;
                    kb1[rr >> 1] = pack_bf16(kbar1, 0.f) & 0xffffu;
                }
            }
            {   // Kbar rows 2pc, 2pc+1 of B2 (N = key channel, K = chunk row)
                unsigned char* b2 = ob + kB2;
                const int c0 = 2 * pc, c1 = 2 * pc + 1;
                *reinterpret_cast<uint4*>(b2 + (c0 >> 3) * kSboB2 + hr * kLbo + (c0 & 7) * 16) =
                    make_uint4(kb0[0], kb0[1], kb0[2], kb0[3]);
                *reinterpret_cast<uint4*>(b2 + (c1 >> 3) * kSboB2 + hr * kLbo + (c1 & 7) * 16) =
                    make_uint4(kb1[0], kb1[1], kb1[2], kb1[3]);
            }
            named_bar_sync(kNamedK1, 128);
            if (kt == 0) mbar_arrive(bar(BAR_IN_EMPTY + s));  // input tiles consumed

            // Phase 2: in-chunk Grams (warp 0: A and the WY solve; warp 1: Mq),
            // warps 2-3 move Qtil into rows 16..31 of B1.
            if (kw < 2) {
                const uint32_t abase = smem_u32(st + (kw == 0 ? ST_KQ : ST_QQ) * kStArr);
                const uint32_t bbase = smem_u32(st + ST_KK * kStArr);
                float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
                for (int k0 = 0; k0 < 128; k0 += 16) {
                    uint32_t a0, a1, a2, a3, b0, b1, b2, b3;
                    ldsm_x4(abase + (lane & 15) * kStRow + (k0 + 8 * (lane >> 4)) * 2, a0, a1, a2, a3);
                    ldsm_x4(bbase + ((lane & 7) + 8 * (lane >> 4)) * kStRow +
                                (k0 + 8 * ((lane >> 3) & 1)) * 2,
                            b0, b1, b2, b3);
                    mma_16816(acc[0], a0, a1, a2, a3, b0, b1);
                    mma_16816(acc[1], a0, a1, a2, a3, b2, b3);
                }
                const int g = lane >> 2, t = lane & 3;
                if (kw == 0) {
#pragma unroll
                    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int r = g + 8 * (e >> 1), sc = 8 * nt + 2 * t + (e & 1);
                            Asm[r * 16 + sc] = sc < r ? bet[r] * acc[nt][e] : 0.f;
                        }
                    __syncwarp();
                    if (lane < 16) {
                        const int sc = lane;
                        float x[kChunk];
#pragma unroll
                        for (int r = 0; r < kChunk; ++r) x[r] = (r == sc) ? 1.f : 0.f;
#pragma unroll
                        for (int m = 0; m < kChunk - 1; ++m)
#pragma unroll
                            for (int r = m + 1; r < kChunk; ++r)
                                x[r] = fmaf(-Asm[r * 16 + m], x[m], x[r]);
                        const float bs = bet[sc];
#pragma unroll
                        for (int r = 0; r < kChunk; ++r) Tb[r * 24 + sc] = __float2bfloat16_rn(x[r] * bs);
                    }
                } else {
                    unsigned char* b3 = ob + kB3;
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
            } else {
                const int ct = kt - 64;  // 0..63
                unsigned char* b1 = ob + kB1;
#pragma unroll
                for (int e = ct; e < 256; e += 64) {
                    const int r = e >> 4, kg = e & 15;
                    *reinterpret_cast<uint4*>(b1 + b1_off(16 + r, kg * 8)) =
                        *reinterpret_cast<const uint4*>(st + ST_QT * kStArr + r * kStRow + kg * 16);
                }
            }
            named_bar_sync(kNamedK1, 128);

            // Phase 3: W = Tb Ktil, U = Tb V; K1 warp kw owns columns [32kw, 32kw + 32).
            {
                uint32_t a0, a1, a2, a3;
                ldsm_x4(smem_u32(Tb) + (lane & 15) * 48 + 8 * (lane >> 4) * 2, a0, a1, a2, a3);
                const int g = lane >> 2, t = lane & 3;
                unsigned char* b1 = ob + kB1;
                float* U = reinterpret_cast<float*>(ob + kU);
#pragma unroll
                for (int which = 0; which < 2; ++which) {
                    const uint32_t bb = smem_u32(st + (which == 0 ? ST_KT : ST_VV) * kStArr);
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
                                *reinterpret_cast<uint32_t*>(b1 + b1_off(g, col)) = pack_bf16(d[0], d[1]);
                                *reinterpret_cast<uint32_t*>(b1 + b1_off(g + 8, col)) = pack_bf16(d[2], d[3]);
                            } else {
                                *reinterpret_cast<float2*>(U + g * 128 + col) = make_float2(d[0], d[1]);
                                *reinterpret_cast<float2*>(U + (g + 8) * 128 + col) = make_float2(d[2], d[3]);
                            }
                        }
                    }
                }
            }
            fence_proxy_async_smem();
            mbar_arrive(bar(BAR_K1_FULL + ks));
        }
    } else {
        // ------------------------------------------------------------ K2 epilogue (256 threads)
        const int quad = warp & 3;
        const int hf = (warp - 6) >> 2;            // 0: key columns 0-63, 1: 64-127
        const int j = 32 * quad + lane;            // value column owned by this thread
        const uint32_t lanes = (uint32_t)(32 * quad) << 16;
        const uint32_t tS = tmem + lanes + kColS + 64u * hf;
        const uint32_t tSA = tmem + lanes + kColSA + 32u * hf;
        const uint32_t tDA = tmem + lanes + kColDA + 4u * hf;
        const size_t soff = ((size_t)n * p.H + h) * kD * kD;
        uint32_t sreg[64];
        // Initial state S0[i][j] for keys i of this half -> S^T[j][i].
#pragma unroll
        for (int i = 0; i < 64; ++i)
            sreg[i] = p.s0 ? __float_as_uint(p.s0[soff + (size_t)(64 * hf + i) * kD + j]) : 0u;
        tmem_st32(tS, sreg);
        tmem_st32(tS + 32, sreg + 32);
        tmem_wait_st();
        bool ok = true;
        int c = 0;
        for (; c < nchunks; ++c) {
            const int ks = c & 1;
            if (c > 0) {
                if (!mbar_wait(bar(BAR_SDONE), (c - 1) & 1, lim)) { ok = false; break; }
                tc_fence_after();
            }
            // (A) S_c (this half) -> bf16 copy for MMA1
            tmem_ld32(tS, sreg);
            tmem_ld32(tS + 32, sreg + 32);
            tmem_wait_ld_regs<64>(sreg);
            {
                uint32_t pk[32];
#pragma unroll
                for (int i = 0; i < 32; ++i)
                    pk[i] = pack_bf16(__uint_as_float(sreg[2 * i]), __uint_as_float(sreg[2 * i + 1]));
                tmem_st32(tSA, pk);
                tmem_wait_st();
            }
            tc_fence_before();
            mbar_arrive(bar(BAR_SA));
            // (C) output rows of the previous chunk, then release its K1 stage
            if (c > 0) {
                const int cp = c - 1;
                const int64_t t0p = bos + (int64_t)cp * kChunk;
                const int Cp = (eos - t0p < kChunk) ? (int)(eos - t0p) : kChunk;
                uint32_t o[8];
                tmem_ld8(tmem + lanes + kColD1 + 32u * (cp & 1) + 16 + 8 * hf, o);
                tmem_wait_ld_regs<8>(o);
#pragma unroll
                for (int r = 0; r < 8; ++r) {
                    const int row = 8 * hf + r;
                    if (row < Cp)
                        p.out[((t0p + row) * H + h) * kD + j] =
                            __float2bfloat16_rn(p.scale * __uint_as_float(o[r]));
                }
                mbar_arrive(bar(BAR_K1_EMPTY + (cp & 1)));
            }
            // (D) decay S by exp(gam_C) ahead of MMA2
            if (!mbar_wait(bar(BAR_K1_FULL + ks), (c >> 1) & 1, lim)) { ok = false; break; }
            const unsigned char* ob = smem + kSmOut + ks * kOutBytes;
            {
                const float4* gc4 = reinterpret_cast<const float4*>(ob + kGC) + 16 * hf;
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
            }
            // (B) delta^T = U^T - (S^T W^T) for rows 8hf .. 8hf+7
            if (!mbar_wait(bar(BAR_D1), c & 1, lim)) { ok = false; break; }
            tc_fence_after();
            {
                uint32_t d[8];
                tmem_ld8(tmem + lanes + kColD1 + 32u * (c & 1) + 8 * hf, d);
                tmem_wait_ld_regs<8>(d);
                const float* U = reinterpret_cast<const float*>(ob + kU);
                uint32_t pk[4];
#pragma unroll
                for (int r = 0; r < 4; ++r) {
                    const int r0 = 8 * hf + 2 * r;
                    const float d0 = U[r0 * 128 + j] - __uint_as_float(d[2 * r]);
                    const float d1 = U[(r0 + 1) * 128 + j] - __uint_as_float(d[2 * r + 1]);
                    pk[r] = pack_bf16(d0, d1);
                }
                tmem_st4(tDA, pk);
                tmem_wait_st();
            }
            tc_fence_before();
            mbar_arrive(bar(BAR_DL));
        }
        if (ok && nchunks > 0) {
            // Output of the last chunk and the final state.
            if (!mbar_wait(bar(BAR_SDONE), (nchunks - 1) & 1, lim)) {
                ok = false;
            } else {
                tc_fence_after();
                const int cp = nchunks - 1;
                const int64_t t0p = bos + (int64_t)cp * kChunk;
                const int Cp = (eos - t0p < kChunk) ? (int)(eos - t0p) : kChunk;
                uint32_t o[8];
                tmem_ld8(tmem + lanes + kColD1 + 32u * (cp & 1) + 16 + 8 * hf, o);
                tmem_wait_ld_regs<8>(o);
#pragma unroll
                for (int r = 0; r < 8; ++r) {
                    const int row = 8 * hf + r;
                    if (row < Cp)
                        p.out[((t0p + row) * H + h) * kD + j] =
                            __float2bfloat16_rn(p.scale * __uint_as_float(o[r]));
                }
            }
        }
        if (!ok) {
            record(p.status, kStatusTimeout);
            tmem_wait_st();
            tmem_wait_ld();
        } else if (p.sfin) {
            tmem_ld32(tS, sreg);
            tmem_ld32(tS + 32, sreg + 32);
            tmem_wait_ld_regs<64>(sreg);
#pragma unroll
            for (int i = 0; i < 64; ++i)
                p.sfin[soff + (size_t)(64 * hf + i) * kD + j] = __uint_as_float(sreg[i]);
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

}  // namespace

size_t serial_smem_bytes() { return kSmemBytes; }
const void* serial_kernel_symbol() { return reinterpret_cast<const void*>(&kda_fwd_tc_kernel); }

cudaError_t launch_serial(const FwdParams& p, const TensorMaps& maps, cudaStream_t stream) {
    const long long blocks = (long long)p.N * p.H;
    if (blocks == 0) return cudaSuccess;
    kda_fwd_tc_kernel<<<(unsigned)blocks, kThreads, kSmemBytes, stream>>>(maps.q, maps.k, maps.v,
                                                                          maps.g, p);
    return cudaGetLastError();
}

}  // namespace kda
