// kda_api.cu -- the C ABI (include/kda.h): validation, device cache, workspaces,
// launch and status reporting.  Host code only; the kernels live in their own
// translation units and are reached through kda_internal.cuh.
//
// Conventions follow the pages' reviews of the reference bindings: per-device
// queries are cached instead of repeated on every launch (flashinfer PR #4313,
// review of the FlashKDA binding's per-launch capability checks); scratch is
// keyed by (device, stream) so concurrent streams never share it and is
// bounded (cuLA PR #103, review of the "_get_scratch" cache); an exact alias of
// the initial and final state is allowed for in-place updates, any partial
// overlap is rejected (flashinfer PR #4351, review of the overlap checks).
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <memory>
#include <mutex>
#include <vector>

#include "../../include/kda.h"
#include "kda_internal.cuh"

namespace {

thread_local char t_last_error[512] = "";

kda_status fail(kda_status st, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(t_last_error, sizeof(t_last_error), fmt, ap);
    va_end(ap);
    return st;
}

kda_status cuda_fail(cudaError_t e, const char* what) {
    return fail(KDA_ERR_CUDA, "%s failed: %s", what, cudaGetErrorString(e));
}

__device__ int32_t g_status_word = 0;

constexpr int kMaxDevices = 64;
constexpr int64_t kDefaultWaitLimit = 1ll << 22;
constexpr size_t kMaxWorkspaces = 8;
constexpr int kMaxHostPieces = 64;  // pieces kda_prefill_host may stream a call in

struct DeviceInfo {
    bool ready = false;
    int cc_major = 0, cc_minor = 0, sm_count = 0;
    int resident_clusters = 0;  // co-resident 2-CTA clusters of the fused kernel
    int32_t* status = nullptr;
};

std::mutex g_mutex;
DeviceInfo g_devices[kMaxDevices];

kda_status device_info(int dev, DeviceInfo** out) {
    if (dev < 0 || dev >= kMaxDevices) return fail(KDA_ERR_UNSUPPORTED_DEVICE, "device %d", dev);
    std::lock_guard<std::mutex> lock(g_mutex);
    DeviceInfo& d = g_devices[dev];
    if (!d.ready) {
        cudaError_t e;
        if ((e = cudaDeviceGetAttribute(&d.cc_major, cudaDevAttrComputeCapabilityMajor, dev)) ||
            (e = cudaDeviceGetAttribute(&d.cc_minor, cudaDevAttrComputeCapabilityMinor, dev)) ||
            (e = cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev)))
            return cuda_fail(e, "cudaDeviceGetAttribute");
        if (d.cc_major != 10 || d.cc_minor != 3)
            return fail(KDA_ERR_UNSUPPORTED_DEVICE,
                        "device %d has compute capability %d.%d; this library is built for "
                        "sm_103a (10.3) only", dev, d.cc_major, d.cc_minor);
        if ((e = cudaGetSymbolAddress(reinterpret_cast<void**>(&d.status), g_status_word)))
            return cuda_fail(e, "cudaGetSymbolAddress(status word)");
        if ((e = cudaFuncSetAttribute(kda::serial_kernel_symbol(),
                                      cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      (int)kda::serial_smem_bytes())))
            return cuda_fail(e, "cudaFuncSetAttribute(serial kernel)");
        if ((e = cudaFuncSetAttribute(kda::grouped_kernel_symbol(),
                                      cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      (int)kda::serial_smem_bytes())))
            return cuda_fail(e, "cudaFuncSetAttribute(grouped kernel)");
        if ((e = kda::merge_init())) return cuda_fail(e, "cudaFuncSetAttribute(merge kernels)");
        {
            cudaLaunchConfig_t cfg = {};
            cfg.gridDim = dim3(2, 1, 1);
            cfg.blockDim = dim3(kda::serial_block_threads(), 1, 1);
            cfg.dynamicSmemBytes = kda::serial_smem_bytes();
            cudaLaunchAttribute attr[1];
            attr[0].id = cudaLaunchAttributeClusterDimension;
            attr[0].val.clusterDim.x = 2;
            attr[0].val.clusterDim.y = 1;
            attr[0].val.clusterDim.z = 1;
            cfg.attrs = attr;
            cfg.numAttrs = 1;
            int n = 0;
            if (cudaOccupancyMaxActiveClusters(&n, kda::serial_kernel_symbol(), &cfg) != cudaSuccess ||
                n < 1) {
                cudaGetLastError();  // clear; fall back to one cluster per SM pair
                n = d.sm_count / 2;
            }
            d.resident_clusters = n > 0 ? n : 1;
        }
        d.ready = true;
    }
    *out = &d;
    return KDA_OK;
}

// ---------------------------------------------------------------------------
// Workspaces: one device buffer per (device, stream), grown on demand, at most
// kMaxWorkspaces alive (least recently used evicted).
enum WorkspaceKind { kWsSegment = 0, kWsHostArena = 1 };

struct Workspace {
    int device;
    void* stream;
    int kind;
    void* ptr;
    size_t bytes;
    unsigned long long last_use;
};
std::vector<Workspace> g_workspaces;
unsigned long long g_use_clock = 0;

kda_status get_workspace(int dev, cudaStream_t stream, int kind, size_t bytes, void** out) {
    *out = nullptr;
    if (bytes == 0) return KDA_OK;
    std::lock_guard<std::mutex> lock(g_mutex);
    for (auto& w : g_workspaces)
        if (w.device == dev && w.stream == (void*)stream && w.kind == kind && w.bytes >= bytes) {
            w.last_use = ++g_use_clock;
            *out = w.ptr;
            return KDA_OK;
        }
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(stream, &cap) == cudaSuccess && cap != cudaStreamCaptureStatusNone)
        return fail(KDA_ERR_CAPTURE_NEEDS_WARMUP,
                    "a %zu-byte workspace is needed while the stream is being captured; run "
                    "the same call once before capture", bytes);
    // Replace a smaller buffer of the same key, else evict the LRU entry when full.
    for (size_t i = 0; i < g_workspaces.size(); ++i)
        if (g_workspaces[i].device == dev && g_workspaces[i].stream == (void*)stream &&
            g_workspaces[i].kind == kind) {
            cudaStreamSynchronize(stream);
            cudaFree(g_workspaces[i].ptr);
            g_workspaces.erase(g_workspaces.begin() + i);
            break;
        }
    if (g_workspaces.size() >= kMaxWorkspaces) {
        size_t lru = 0;
        for (size_t i = 1; i < g_workspaces.size(); ++i)
            if (g_workspaces[i].last_use < g_workspaces[lru].last_use) lru = i;
        int cur;
        cudaGetDevice(&cur);
        cudaSetDevice(g_workspaces[lru].device);
        cudaDeviceSynchronize();
        cudaFree(g_workspaces[lru].ptr);
        cudaSetDevice(cur);
        g_workspaces.erase(g_workspaces.begin() + lru);
    }
    void* p = nullptr;
    cudaError_t e = cudaMalloc(&p, bytes);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return fail(KDA_ERR_OUT_OF_MEMORY, "cudaMalloc(%zu) for a workspace failed: %s", bytes,
                    cudaGetErrorString(e));
    }
    g_workspaces.push_back({dev, (void*)stream, kind, p, bytes, ++g_use_clock});
    *out = p;
    return KDA_OK;
}

// ---------------------------------------------------------------------------
// TMA descriptors.  cuTensorMapEncodeTiled is reached through the runtime's
// driver entry-point query, so the library does not link libcuda directly.
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

kda_status encoder(PFN_cuTensorMapEncodeTiled_v12000* fn) {
    std::lock_guard<std::mutex> lock(g_mutex);
    if (!g_encode) {
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        void* f = nullptr;
        cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000,
                                                         cudaEnableDefault, &q);
        if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !f)
            return fail(KDA_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable (%s)",
                        cudaGetErrorString(e));
        g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    }
    *fn = g_encode;
    return KDA_OK;
}

// [T][H][128] tensor of `elem` bytes per element; box = one 16-row chunk of one head.
kda_status encode_chunk_map(CUtensorMap* m, const void* base, CUtensorMapDataType dt, int elem,
                            int64_t T, int32_t H, const char* name) {
    PFN_cuTensorMapEncodeTiled_v12000 fn;
    kda_status st = encoder(&fn);
    if (st != KDA_OK) return st;
    cuuint64_t dims[3] = {(cuuint64_t)kda::kD, (cuuint64_t)H, (cuuint64_t)T};
    cuuint64_t strides[2] = {(cuuint64_t)kda::kD * elem, (cuuint64_t)H * kda::kD * elem};
    cuuint32_t box[3] = {(cuuint32_t)kda::kD, 1, (cuuint32_t)kda::kChunk};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(m, dt, 3, const_cast<void*>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return fail(KDA_ERR_CUDA, "cuTensorMapEncodeTiled(%s) failed with CUresult %d", name,
                    (int)r);
    return KDA_OK;
}

// ---------------------------------------------------------------------------
struct Range {
    const void* p;
    size_t bytes;
};

bool overlaps(Range a, Range b) {
    if (!a.p || !b.p || a.bytes == 0 || b.bytes == 0) return false;
    const uintptr_t a0 = (uintptr_t)a.p, b0 = (uintptr_t)b.p;
    return a0 < b0 + b.bytes && b0 < a0 + a.bytes;
}

bool aligned(const void* p, size_t a) { return ((uintptr_t)p % a) == 0; }

struct Problem {
    int64_t T_total, dense_len;
    int32_t N, H;        // H: heads of v, g, beta and the states
    int32_t Hq, Hk, Ho;  // heads of q, of k (min(Hq, H)) and of the output (max(Hq, H))
    bool varlen;
};

// Bytes of each tensor of a problem (states in elements of `state_elem` bytes).
struct Sizes {
    size_t q, k, v, g, beta, out, state;
};
Sizes sizes_of(const Problem& pr, size_t state_elem = 4) {
    const size_t t = (size_t)pr.T_total * kda::kD;
    return {t * pr.Hq * 2, t * pr.Hk * 2, t * pr.H * 2, t * pr.H * 4, (size_t)pr.T_total * pr.H * 2,
            t * pr.Ho * 2, (size_t)pr.N * pr.H * kda::kD * kda::kD * state_elem};
}

kda_status validate_shape(const kda_shape* s, bool varlen, Problem* pr) {
    if (!s) return fail(KDA_ERR_INVALID_ARGUMENT, "shape is NULL");
    if (s->head_dim != kda::kD)
        return fail(KDA_ERR_INVALID_ARGUMENT, "head_dim must be 128 (got %d)", s->head_dim);
    if (s->num_heads <= 0)
        return fail(KDA_ERR_INVALID_ARGUMENT, "num_heads must be >= 1 (got %d)", s->num_heads);
    if (s->seq_len < 0)
        return fail(KDA_ERR_INVALID_ARGUMENT, "seq_len must be >= 0 (got %lld)",
                    (long long)s->seq_len);
    pr->H = s->num_heads;
    pr->Hq = s->num_q_heads ? s->num_q_heads : s->num_heads;
    if (pr->Hq < 0 || (pr->Hq % pr->H != 0 && pr->H % pr->Hq != 0))
        return fail(KDA_ERR_INVALID_ARGUMENT,
                    "num_q_heads (%d) and num_heads (%d) must divide one another",
                    s->num_q_heads, s->num_heads);
    pr->Hk = pr->Hq < pr->H ? pr->Hq : pr->H;
    pr->Ho = pr->Hq > pr->H ? pr->Hq : pr->H;
    pr->varlen = varlen;
    if (varlen) {
        if (s->batch != 1)
            return fail(KDA_ERR_INVALID_ARGUMENT, "packed varlen input needs batch == 1 (got %d)",
                        s->batch);
        if (s->num_seqs <= 0)
            return fail(KDA_ERR_INVALID_ARGUMENT, "num_seqs must be >= 1 with cu_seqlens (got %d)",
                        s->num_seqs);
        pr->N = s->num_seqs;
        pr->T_total = s->seq_len;
        pr->dense_len = 0;
    } else {
        if (s->batch <= 0)
            return fail(KDA_ERR_INVALID_ARGUMENT, "batch must be >= 1 (got %d)", s->batch);
        pr->N = s->batch;
        pr->dense_len = s->seq_len;
        if (s->seq_len > (int64_t)1 << 40)
            return fail(KDA_ERR_INVALID_ARGUMENT, "seq_len too large");
        pr->T_total = (int64_t)s->batch * s->seq_len;
    }
    if ((int64_t)pr->N * pr->Ho > 0x3fffffffll)
        return fail(KDA_ERR_INVALID_ARGUMENT, "num_seqs * max(num_heads, num_q_heads) exceeds 2^30 - 1");
    if (pr->T_total > ((int64_t)1 << 46) / ((int64_t)pr->Ho * kda::kD))
        return fail(KDA_ERR_INVALID_ARGUMENT, "T_total * heads * 128 is too large");
    return KDA_OK;
}

kda_status validate_options(const kda_options* o, const Problem& pr, int32_t* mode,
                            int32_t* seg_len, int64_t* wait_limit, int32_t* debug_flags,
                            int32_t* state_bf16 = nullptr) {
    *mode = KDA_MODE_SERIAL;
    *seg_len = 8192;
    *wait_limit = kDefaultWaitLimit;
    *debug_flags = 0;
    if (state_bf16) *state_bf16 = 0;
    if (!o) return KDA_OK;
    if (o->state_dtype != KDA_STATE_F32 && o->state_dtype != KDA_STATE_BF16)
        return fail(KDA_ERR_INVALID_ARGUMENT, "unknown state_dtype %d", o->state_dtype);
    if (state_bf16) *state_bf16 = o->state_dtype == KDA_STATE_BF16;
    if (o->debug_flags & ~KDA_DEBUG_STALL_WAIT)
        return fail(KDA_ERR_INVALID_ARGUMENT, "unknown debug_flags bits 0x%x", o->debug_flags);
    if (o->host_pieces < 0 || o->host_pieces > kMaxHostPieces)
        return fail(KDA_ERR_INVALID_ARGUMENT, "host_pieces must be in [0, %d] (got %d)",
                    kMaxHostPieces, o->host_pieces);
    *debug_flags = o->debug_flags;
    if (o->mode != KDA_MODE_SERIAL && o->mode != KDA_MODE_SEGMENT && o->mode != KDA_MODE_AUTO)
        return fail(KDA_ERR_INVALID_ARGUMENT, "unknown mode %d", o->mode);
    if (o->segment_len < 0 || (o->segment_len % kda::kChunk) != 0)
        return fail(KDA_ERR_INVALID_ARGUMENT,
                    "segment_len must be a non-negative multiple of 16 (got %d)", o->segment_len);
    if (o->wait_limit < 0)
        return fail(KDA_ERR_INVALID_ARGUMENT, "wait_limit must be >= 0");
    *mode = o->mode;
    if (o->segment_len) *seg_len = o->segment_len;
    if (o->wait_limit) *wait_limit = o->wait_limit;
    return KDA_OK;
}

kda_status validate_pointers(const Problem& pr, const uint16_t* q, const uint16_t* k,
                             const uint16_t* v, const float* g, const uint16_t* beta, float scale,
                             const void* s0, const int32_t* cu, const uint16_t* out,
                             const void* sfin, size_t state_elem = 4) {
    if (!(scale == scale) || scale > 3.4e38f || scale < -3.4e38f)
        return fail(KDA_ERR_INVALID_ARGUMENT, "scale must be finite");
    const Sizes sz = sizes_of(pr, state_elem);
    const size_t cub = pr.varlen ? (size_t)(pr.N + 1) * 4 : 0;
    if (pr.T_total > 0) {
        const void* req[] = {q, k, v, g, beta, out};
        const char* names[] = {"q", "k", "v", "g", "beta", "out"};
        for (int i = 0; i < 6; ++i)
            if (!req[i]) return fail(KDA_ERR_INVALID_ARGUMENT, "%s is NULL", names[i]);
        const void* al16[] = {q, k, v, g, out};
        const char* n16[] = {"q", "k", "v", "g", "out"};
        for (int i = 0; i < 5; ++i)
            if (!aligned(al16[i], 16))
                return fail(KDA_ERR_INVALID_ARGUMENT, "%s must be 16-byte aligned", n16[i]);
        if (!aligned(beta, 2)) return fail(KDA_ERR_INVALID_ARGUMENT, "beta must be 2-byte aligned");
    }
    if (pr.varlen && !cu) return fail(KDA_ERR_INVALID_ARGUMENT, "cu_seqlens is NULL");
    if (cu && !aligned(cu, 4)) return fail(KDA_ERR_INVALID_ARGUMENT, "cu_seqlens must be 4-byte aligned");
    if (s0 && !aligned(s0, 16))
        return fail(KDA_ERR_INVALID_ARGUMENT, "initial_state must be 16-byte aligned");
    if (sfin && !aligned(sfin, 16))
        return fail(KDA_ERR_INVALID_ARGUMENT, "final_state must be 16-byte aligned");

    const Range rq{q, sz.q}, rk{k, sz.k}, rv{v, sz.v}, rg{g, sz.g}, rb{beta, sz.beta},
        rs0{s0, sz.state}, rcu{cu, cub}, rout{out, sz.out}, rfin{sfin, sz.state};
    const Range ins[] = {rq, rk, rv, rg, rb, rs0, rcu, rfin};
    const char* in_names[] = {"q", "k", "v", "g", "beta", "initial_state", "cu_seqlens",
                              "final_state"};
    for (int i = 0; i < 8; ++i)
        if (overlaps(rout, ins[i]))
            return fail(KDA_ERR_ALIASING, "out overlaps %s", in_names[i]);
    const Range fin_ins[] = {rq, rk, rv, rg, rb, rcu};
    for (int i = 0; i < 6; ++i)
        if (overlaps(rfin, fin_ins[i]))
            return fail(KDA_ERR_ALIASING, "final_state overlaps %s", in_names[i]);
    if (s0 && sfin && s0 != sfin && overlaps(rs0, rfin))
        return fail(KDA_ERR_ALIASING,
                    "initial_state and final_state overlap without being the same buffer");
    return KDA_OK;
}

// Segment-mode plan: number of segments per sequence and workspace layout
// (b_seg, m_seg: [B][nseg-1][H][128][128]; carries: [B][nseg][H][128][128], fp32).
struct SegPlan {
    int32_t nseg = 0;
    size_t off_b = 0, off_m = 0, off_c = 0, bytes = 0;
};

// Serial or segment mode, and the segment length, for a problem with `resident`
// co-resident clusters.  Cost unit: one chunk period of one state chain.  Every pass of
// the fused kernel (serial; segment summary, transition and output passes) costs about
// the same per chunk on GB300 (T = 131072: serial 0.82 us per chunk with 4 heads and
// 0.88 us with 64, the segment passes 0.82 and 0.85 us per chunk of the busiest cluster
// slot), clusters beyond `resident` run in further waves, and each segment adds a fixed
// cost (the merge walks a chain's segments one after another; each short cluster fills
// its pipeline).  Fitted on GB300 from T = 131072, H = 4 with segments of 512 .. 16384
// tokens (1.32 .. 2.54 ms against 6.70 ms serial): about 5 chunk periods per segment,
// within 3% at every point.
constexpr double kMergePerSegment = 5.0;
constexpr double kSegmentMargin = 0.8;      // segment mode must win by 20%
constexpr size_t kPlanWorkspaceCap = (size_t)4 << 30;
constexpr int64_t kMinPlanSegment = 512;  // shortest segment the planner considers

void choose_plan(const Problem& pr, int64_t resident, int32_t* mode, int32_t* seg_len) {
    *mode = KDA_MODE_SERIAL;
    *seg_len = 0;
    if (pr.varlen || pr.dense_len <= 0) return;
    // Chains of the summary passes (one per state head) and of the output pass (one per
    // output head; more with grouped query heads).
    const int64_t C = (int64_t)pr.N * pr.H, Co = (int64_t)pr.N * pr.Ho;
    const int64_t R = resident > 0 ? resident : 1;
    auto cdiv = [](int64_t a, int64_t b) { return (a + b - 1) / b; };
    const int64_t nck = cdiv(pr.dense_len, kda::kChunk);
    const double serial = (double)cdiv(Co, R) * (double)nck;
    double best = serial;
    int32_t best_len = 0;
    // Candidates: for each segment count n, the shortest multiple of 16 tokens that covers
    // the sequence in n segments.  These include every count whose passes fill the cluster
    // slots exactly (C n = R for few chains), which lengths on a power-of-two grid miss.
    int64_t prev = -1;
    for (int64_t n = 2;; ++n) {
        const int64_t sl = cdiv(cdiv(pr.dense_len, n), kda::kChunk) * kda::kChunk;
        if (sl < kMinPlanSegment) break;
        if (sl == prev || sl > ((int64_t)1 << 30)) continue;
        prev = sl;
        const int64_t nseg = cdiv(pr.dense_len, sl);
        const size_t ws = (size_t)(3 * nseg - 2) * (size_t)C * kda::kD * kda::kD * 4;
        if (ws > kPlanWorkspaceCap) break;  // grows with n
        const double waves = (double)(2 * cdiv(C * (nseg - 1), R) + cdiv(Co * nseg, R));
        const double cost = waves * (double)(sl / kda::kChunk) + kMergePerSegment * (double)nseg;
        if (cost < best) {
            best = cost;
            best_len = (int32_t)sl;
        }
    }
    if (best_len && best < kSegmentMargin * serial) {
        *mode = KDA_MODE_SEGMENT;
        *seg_len = best_len;
    }
}

// Packed varlen input whose offsets the host holds (kda_prefill_host, kda_plan_varlen).
// Same units as choose_plan: serial costs the longer of the longest chain and the
// chains' total over the R slots; a segment plan of length L gives sequence n
// max(1, ceil(len_n / L)) rows, its summary and transition passes run every row but each
// sequence's last, its output pass every row, each pass in waves of R rows of at most
// L / 16 chunks, and the merge walks the longest sequence's rows in order.  Candidates:
// for every count n of segments of the longest sequence, the shortest multiple of 16
// tokens covering it in n segments (at least 512).
void choose_plan_varlen(const Problem& pr, const int32_t* cu, int64_t resident, int32_t* mode,
                        int32_t* seg_len) {
    *mode = KDA_MODE_SERIAL;
    *seg_len = 0;
    const int64_t R = resident > 0 ? resident : 1;
    auto cdiv = [](int64_t a, int64_t b) { return (a + b - 1) / b; };
    int64_t maxlen = 0, total_ck = 0, max_ck = 0;
    for (int n = 0; n < pr.N; ++n) {
        const int64_t len = (int64_t)cu[n + 1] - cu[n];
        maxlen = len > maxlen ? len : maxlen;
        total_ck += cdiv(len, kda::kChunk);
        max_ck = cdiv(len, kda::kChunk) > max_ck ? cdiv(len, kda::kChunk) : max_ck;
    }
    const double serial = (double)std::max(max_ck, cdiv(total_ck * pr.Ho, R));
    double best = serial;
    int32_t best_len = 0;
    int64_t prev = -1;
    for (int64_t n = 2;; ++n) {
        const int64_t sl = cdiv(cdiv(maxlen, n), kda::kChunk) * kda::kChunk;
        if (sl < kMinPlanSegment) break;
        if (sl == prev || sl > ((int64_t)1 << 30) || sl >= pr.T_total) continue;
        prev = sl;
        const size_t ws = (size_t)3 * (size_t)(pr.N + pr.T_total / sl) * pr.H * kda::kD * kda::kD * 4;
        if (ws > kPlanWorkspaceCap) break;  // grows with n
        int64_t rows = 0, inner = 0, max_rows = 0;
        for (int i = 0; i < pr.N; ++i) {
            const int64_t len = (int64_t)cu[i + 1] - cu[i];
            const int64_t r = len > 0 ? cdiv(len, sl) : 1;
            rows += r;
            inner += r - 1;
            max_rows = r > max_rows ? r : max_rows;
        }
        const int64_t l = sl / kda::kChunk;
        const double cost = (inner > 0 ? 2.0 * (double)cdiv(inner * pr.H, R) * (double)l : 0.0) +
                            (double)cdiv(rows * pr.Ho, R) * (double)l + kMergePerSegment * (double)max_rows;
        if (cost < best) {
            best = cost;
            best_len = (int32_t)sl;
        }
    }
    if (best_len && best < kSegmentMargin * serial) {
        *mode = KDA_MODE_SEGMENT;
        *seg_len = best_len;
    }
}

// Query heads a segment summary pass is launched with: summaries and transitions write
// no output, so one cluster per state head does (with grouped query heads, the equal-count
// instance, whose state head h reads k head h and an unused q head).
int32_t summary_q_heads(const Problem& pr) { return pr.Hq > pr.H ? pr.H : pr.Hq; }

// Varlen segment plan: sequence n gets max(1, ceil(len_n / seg_len)) segments, at most
// N + floor(T_total / seg_len) in all; the table, summaries, transitions and carries are
// sized for that bound (rows past the actual count exit at once).
struct VarSegPlan {
    int64_t rows = 0;  // 0: serial
    size_t off_tab = 0, off_b = 0, off_m = 0, off_c = 0, bytes = 0;
};

VarSegPlan plan_segments_varlen(const Problem& pr, int32_t seg_len) {
    VarSegPlan vp;
    if (!pr.varlen || seg_len <= 0 || pr.T_total <= seg_len) return vp;
    vp.rows = (int64_t)pr.N + pr.T_total / seg_len;
    const size_t st = (size_t)kda::kD * kda::kD * 4;
    const size_t per = (size_t)vp.rows * pr.H * st;
    vp.off_tab = 0;
    vp.off_b = ((size_t)(pr.N + 1) * 4 + 255) / 256 * 256;
    vp.off_m = vp.off_b + per;
    vp.off_c = vp.off_m + per;
    vp.bytes = vp.off_c + per;
    return vp;
}

SegPlan plan_segments(const Problem& pr, int32_t seg_len) {
    SegPlan sp;
    if (pr.varlen || pr.dense_len <= 0 || seg_len <= 0) return sp;
    sp.nseg = (int32_t)((pr.dense_len + seg_len - 1) / seg_len);
    if (sp.nseg <= 1) return sp;
    const size_t st = (size_t)kda::kD * kda::kD * 4;
    const size_t per = (size_t)pr.N * pr.H * st;
    sp.off_b = 0;
    sp.off_m = per * (sp.nseg - 1);
    sp.off_c = 2 * per * (sp.nseg - 1);
    sp.bytes = sp.off_c + per * sp.nseg;
    return sp;
}

// Kernel parameters of one call (pointers, sizes, wait limit, status word) and the TMA
// descriptors of its tensors; shared by every entry point that launches the prefill.
// s0 / sfin hold fp32 states, or bf16 ones when s0_bf16 / sfin_bf16.
kda_status prepare_call(const Problem& pr, const uint16_t* q, const uint16_t* k, const uint16_t* v,
                        const float* g, const uint16_t* beta, float scale, const void* s0, int32_t s0_bf16,
                        const int32_t* cu, uint16_t* out, void* sfin, int32_t sfin_bf16, int64_t wait_limit,
                        int32_t debug_flags, int32_t* status, kda::FwdParams* p,
                        kda::TensorMaps* maps) {
    *p = kda::FwdParams{};
    p->q = reinterpret_cast<const __nv_bfloat16*>(q);
    p->k = reinterpret_cast<const __nv_bfloat16*>(k);
    p->v = reinterpret_cast<const __nv_bfloat16*>(v);
    p->g = g;
    p->beta = reinterpret_cast<const __nv_bfloat16*>(beta);
    p->s0 = s0;
    p->s0_bf16 = s0 ? s0_bf16 : 0;
    p->sfin = sfin;
    p->sfin_bf16 = sfin ? sfin_bf16 : 0;
    p->out = reinterpret_cast<__nv_bfloat16*>(out);
    p->cu = cu;
    p->T_total = pr.T_total;
    p->dense_len = pr.dense_len;
    p->N = pr.N;
    p->H = pr.H;
    p->Hq = pr.Hq;
    p->scale = scale;
    p->wait_limit = wait_limit;
    p->debug_flags = debug_flags;
    p->status = status;
    memset(maps, 0, sizeof(*maps));
    kda_status st = KDA_OK;
    if (pr.T_total > 0) {
        if ((st = encode_chunk_map(&maps->q, q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, pr.T_total, pr.Hq, "q")) ||
            (st = encode_chunk_map(&maps->k, k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, pr.T_total, pr.Hk, "k")) ||
            (st = encode_chunk_map(&maps->v, v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, pr.T_total, pr.H, "v")) ||
            (st = encode_chunk_map(&maps->g, g, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, pr.T_total, pr.H, "g")) ||
            (st = encode_chunk_map(&maps->out, out, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, pr.T_total, pr.Ho, "out")))
            return st;
    }
    return KDA_OK;
}

// Dense segment-parallel prefill on scratch `base` laid out by `sp` (sp.nseg >= 2):
// pre_scan (segment summaries from zero and transitions from the identity, all segments
// but the last, in parallel) -> merge (carries from the initial state) -> segment-K2.
// Every scratch byte it reads is written earlier in the same call.
kda_status run_dense_segments(const Problem& pr, const kda::FwdParams& p, const kda::TensorMaps& maps,
                              const SegPlan& sp, int32_t seg_len, void* base, int sm_count,
                              cudaStream_t stream) {
    cudaError_t e;
    float* b_seg = reinterpret_cast<float*>(static_cast<char*>(base) + sp.off_b);
    float* m_seg = reinterpret_cast<float*>(static_cast<char*>(base) + sp.off_m);
    float* carries = reinterpret_cast<float*>(static_cast<char*>(base) + sp.off_c);
    kda::FwdParams ps = p;
    ps.Hq = summary_q_heads(pr);
    ps.seg_len = seg_len;
    ps.nseg_total = sp.nseg;
    ps.nseg_used = sp.nseg - 1;
    ps.s0 = nullptr;
    ps.s0_bf16 = 0;
    ps.sfin = b_seg;  // summaries and transitions stay fp32
    ps.sfin_bf16 = 0;
    ps.flags = kda::kFlagNoOutput;
    if ((e = kda::launch_serial(ps, maps, stream)) != cudaSuccess)
        return cuda_fail(e, "pre_scan (summary) launch");
    ps.sfin = m_seg;
    ps.flags = kda::kFlagNoOutput | kda::kFlagZeroV | kda::kFlagIdentityS0;
    if ((e = kda::launch_serial(ps, maps, stream)) != cudaSuccess)
        return cuda_fail(e, "pre_scan (transition) launch");
    if ((e = kda::launch_merge(m_seg, b_seg, p.s0, p.s0_bf16, carries, pr.N, sp.nseg, pr.H, sm_count,
                               stream)) != cudaSuccess)
        return cuda_fail(e, "merge launch");
    kda::FwdParams pk = p;
    pk.seg_len = seg_len;
    pk.nseg_total = sp.nseg;
    pk.nseg_used = sp.nseg;
    pk.s0 = carries;  // fp32; the final state keeps the caller's type
    pk.s0_bf16 = 0;
    pk.flags = kda::kFlagFinalLastSeg;
    if ((e = kda::launch_serial(pk, maps, stream)) != cudaSuccess)
        return cuda_fail(e, "segment-K2 launch");
    return KDA_OK;
}

kda_status run(const Problem& pr, const uint16_t* q, const uint16_t* k, const uint16_t* v,
               const float* g, const uint16_t* beta, float scale, const void* s0, int32_t s0_bf16,
               const int32_t* cu, uint16_t* out, void* sfin, int32_t sfin_bf16, cudaStream_t stream,
               int32_t mode, int32_t seg_len, int64_t wait_limit, int32_t debug_flags) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    DeviceInfo* di = nullptr;
    kda_status st = device_info(dev, &di);
    if (st != KDA_OK) return st;
    if (pr.T_total == 0 && !sfin) return KDA_OK;

    kda::FwdParams p;
    kda::TensorMaps maps;
    if ((st = prepare_call(pr, q, k, v, g, beta, scale, s0, s0_bf16, cu, out, sfin, sfin_bf16, wait_limit,
                           debug_flags, di->status, &p, &maps)) != KDA_OK)
        return st;
    if (mode == KDA_MODE_AUTO) choose_plan(pr, di->resident_clusters, &mode, &seg_len);
    if (mode == KDA_MODE_SEGMENT && pr.varlen) {
        const VarSegPlan vp = plan_segments_varlen(pr, seg_len);
        if (vp.rows > 0) {
            if (vp.rows * 2 * pr.Ho > 0x7fffffffll)
                return fail(KDA_ERR_INVALID_ARGUMENT, "too many segments for one launch");
            // Varlen segments: table -> pre_scan (summaries from zero, transitions from the
            // identity; every segment but each sequence's last) -> merge -> segment-K2.
            void* ws = nullptr;
            if ((st = get_workspace(dev, stream, kWsSegment, vp.bytes, &ws)) != KDA_OK) return st;
            char* base = static_cast<char*>(ws);
            int32_t* table = reinterpret_cast<int32_t*>(base + vp.off_tab);
            float* b_seg = reinterpret_cast<float*>(base + vp.off_b);
            float* m_seg = reinterpret_cast<float*>(base + vp.off_m);
            float* carries = reinterpret_cast<float*>(base + vp.off_c);
            if ((e = kda::launch_segment_table(cu, pr.N, pr.T_total, seg_len, table, di->status,
                                               stream)) != cudaSuccess)
                return cuda_fail(e, "segment table launch");
            kda::FwdParams ps = p;
            ps.Hq = summary_q_heads(pr);
            ps.seg_len = seg_len;
            ps.seg_start = table;
            ps.rows = (int32_t)vp.rows;
            ps.s0 = nullptr;
            ps.s0_bf16 = 0;
            ps.sfin = b_seg;  // summaries and transitions stay fp32
            ps.sfin_bf16 = 0;
            ps.flags = kda::kFlagNoOutput | kda::kFlagSkipLastSeg;
            if ((e = kda::launch_serial(ps, maps, stream)) != cudaSuccess)
                return cuda_fail(e, "pre_scan (summary) launch");
            ps.sfin = m_seg;
            ps.flags = kda::kFlagNoOutput | kda::kFlagZeroV | kda::kFlagIdentityS0 | kda::kFlagSkipLastSeg;
            if ((e = kda::launch_serial(ps, maps, stream)) != cudaSuccess)
                return cuda_fail(e, "pre_scan (transition) launch");
            if ((e = kda::launch_merge(m_seg, b_seg, p.s0, p.s0_bf16, carries, pr.N, 0, pr.H, di->sm_count,
                                      stream, table)) != cudaSuccess)
                return cuda_fail(e, "merge launch");
            kda::FwdParams pk = p;
            pk.seg_len = seg_len;
            pk.seg_start = table;
            pk.rows = (int32_t)vp.rows;
            pk.s0 = carries;  // fp32; the final state keeps the caller's type
            pk.s0_bf16 = 0;
            pk.flags = kda::kFlagFinalLastSeg;
            if ((e = kda::launch_serial(pk, maps, stream)) != cudaSuccess)
                return cuda_fail(e, "segment-K2 launch");
            return KDA_OK;
        }
    }
    const SegPlan sp = mode == KDA_MODE_SEGMENT ? plan_segments(pr, seg_len) : SegPlan{};
    if (sp.nseg <= 1) {
        e = kda::launch_serial(p, maps, stream);
        if (e != cudaSuccess) return cuda_fail(e, "serial prefill launch");
        return KDA_OK;
    }
    void* ws = nullptr;
    if ((st = get_workspace(dev, stream, kWsSegment, sp.bytes, &ws)) != KDA_OK) return st;
    return run_dense_segments(pr, p, maps, sp, seg_len, ws, di->sm_count, stream);
}

}  // namespace

extern "C" {

kda_status kda_prefill_ex(const kda_shape* shape, const uint16_t* q, const uint16_t* k,
                          const uint16_t* v, const float* g, const uint16_t* beta, float scale,
                          const void* initial_state, const int32_t* cu_seqlens, uint16_t* out,
                          void* final_state, void* stream, const kda_options* opts) {
    t_last_error[0] = '\0';
    Problem pr{};
    kda_status st = validate_shape(shape, cu_seqlens != nullptr, &pr);
    if (st != KDA_OK) return st;
    int32_t mode, seg_len, debug_flags, sbf;
    int64_t wait_limit;
    if ((st = validate_options(opts, pr, &mode, &seg_len, &wait_limit, &debug_flags, &sbf)) != KDA_OK)
        return st;
    if ((st = validate_pointers(pr, q, k, v, g, beta, scale, initial_state, cu_seqlens, out,
                                final_state, sbf ? 2 : 4)) != KDA_OK)
        return st;
    return run(pr, q, k, v, g, beta, scale, initial_state, sbf, cu_seqlens, out, final_state, sbf,
               (cudaStream_t)stream, mode, seg_len, wait_limit, debug_flags);
}

kda_status kda_prefill(const kda_shape* shape, const uint16_t* q, const uint16_t* k,
                       const uint16_t* v, const float* g, const uint16_t* beta, float scale,
                       const float* initial_state, const int32_t* cu_seqlens, uint16_t* out,
                       float* final_state, void* stream) {
    return kda_prefill_ex(shape, q, k, v, g, beta, scale, initial_state, cu_seqlens, out,
                          final_state, stream, nullptr);
}

// ---------------------------------------------------------------------------
// kda_prefill_host streams the host buffers through the GPU in pieces: piece b's inputs
// copy in on a copy-in stream while earlier pieces compute on the caller's stream and
// their outputs copy out on a copy-out stream, so the host link carries both directions
// at once and the kernels hide under the copies.  Several sequences split into ranges of
// whole sequences (every chain computes exactly as in one call); one sequence splits into
// token blocks of whole chunks, its fp32 state carried from block to block in place.
constexpr int kAutoHostPieces = 8;
constexpr size_t kHostPipelineMinBytes = (size_t)32 << 20;  // smaller inputs: one piece

struct HostPipe {
    int device = 0;
    void* stream = nullptr;
    cudaStream_t in = nullptr, out = nullptr;  // copy-in and copy-out streams
    cudaEvent_t start = nullptr, out_done = nullptr;
    cudaEvent_t in_done[kMaxHostPieces] = {}, computed[kMaxHostPieces] = {};
    unsigned long long last_use = 0;
};
std::vector<std::unique_ptr<HostPipe>> g_pipes;  // per (device, caller stream), g_mutex

void destroy_pipe(HostPipe& hp) {
    int cur = 0;
    cudaGetDevice(&cur);
    cudaSetDevice(hp.device);
    for (cudaStream_t st : {hp.in, hp.out})
        if (st) {
            cudaStreamSynchronize(st);
            cudaStreamDestroy(st);
        }
    for (cudaEvent_t ev : {hp.start, hp.out_done})
        if (ev) cudaEventDestroy(ev);
    for (int i = 0; i < kMaxHostPieces; ++i) {
        if (hp.in_done[i]) cudaEventDestroy(hp.in_done[i]);
        if (hp.computed[i]) cudaEventDestroy(hp.computed[i]);
    }
    cudaSetDevice(cur);
}

kda_status get_pipe(int dev, cudaStream_t stream, HostPipe** out) {
    std::lock_guard<std::mutex> lock(g_mutex);
    for (auto& hp : g_pipes)
        if (hp->device == dev && hp->stream == (void*)stream) {
            hp->last_use = ++g_use_clock;
            *out = hp.get();
            return KDA_OK;
        }
    if (g_pipes.size() >= kMaxWorkspaces) {
        size_t lru = 0;
        for (size_t i = 1; i < g_pipes.size(); ++i)
            if (g_pipes[i]->last_use < g_pipes[lru]->last_use) lru = i;
        destroy_pipe(*g_pipes[lru]);
        g_pipes.erase(g_pipes.begin() + lru);
    }
    auto hp = std::make_unique<HostPipe>();
    hp->device = dev;
    hp->stream = (void*)stream;
    cudaError_t e;
    const unsigned ef = cudaEventDisableTiming;
    if ((e = cudaStreamCreateWithFlags(&hp->in, cudaStreamNonBlocking)) ||
        (e = cudaStreamCreateWithFlags(&hp->out, cudaStreamNonBlocking)) ||
        (e = cudaEventCreateWithFlags(&hp->start, ef)) ||
        (e = cudaEventCreateWithFlags(&hp->out_done, ef))) {
        destroy_pipe(*hp);
        return cuda_fail(e, "copy stream / event creation");
    }
    for (int i = 0; i < kMaxHostPieces; ++i)
        if ((e = cudaEventCreateWithFlags(&hp->in_done[i], ef)) ||
            (e = cudaEventCreateWithFlags(&hp->computed[i], ef))) {
            destroy_pipe(*hp);
            return cuda_fail(e, "copy event creation");
        }
    hp->last_use = ++g_use_clock;
    *out = hp.get();
    g_pipes.push_back(std::move(hp));
    return KDA_OK;
}

struct HostPiece {
    int32_t n0, n1;  // sequences [n0, n1) (a token block: 0, 1)
    int64_t t0, t1;  // tokens [t0, t1) of the flattened token axis
};

// At most `want` pieces of a problem: balanced ranges of whole sequences when there are
// several, else token blocks of whole chunks of the one sequence (*blocks = true).
std::vector<HostPiece> host_pieces(const Problem& pr, const int32_t* cu, int want, bool* blocks) {
    std::vector<HostPiece> v;
    *blocks = false;
    auto start = [&](int32_t n) -> int64_t { return cu ? (int64_t)cu[n] : (int64_t)n * pr.dense_len; };
    if (want <= 1 || pr.T_total == 0) {
        v.push_back({0, pr.N, 0, pr.T_total});
        return v;
    }
    if (pr.N >= 2) {
        const int P = want < pr.N ? want : pr.N;
        int32_t n0 = 0;
        for (int b = 1; b <= P; ++b) {
            int32_t n1 = pr.N;
            if (b < P) {  // the first sequence end at or past b/P of the tokens, leaving
                          // one sequence at least for every later piece
                const int64_t target = pr.T_total * b / P;
                n1 = n0 + 1;
                while (n1 < pr.N - (P - b) && start(n1) < target) ++n1;
            }
            v.push_back({n0, n1, start(n0), start(n1)});
            n0 = n1;
        }
        return v;
    }
    const int64_t nck = (pr.T_total + kda::kChunk - 1) / kda::kChunk;
    const int64_t P = want < nck ? want : nck;
    const int64_t per = (nck + P - 1) / P * kda::kChunk;
    *blocks = true;
    for (int64_t t0 = 0; t0 < pr.T_total; t0 += per)
        v.push_back({0, 1, t0, t0 + per < pr.T_total ? t0 + per : pr.T_total});
    return v;
}

kda_status kda_prefill_host(const kda_shape* shape, const uint16_t* q, const uint16_t* k,
                            const uint16_t* v, const float* g, const uint16_t* beta,
                            float scale, const void* initial_state,
                            const int32_t* cu_seqlens, uint16_t* out, void* final_state,
                            void* stream_, const kda_options* opts) {
    t_last_error[0] = '\0';
    cudaStream_t stream = (cudaStream_t)stream_;
    Problem pr{};
    kda_status st = validate_shape(shape, cu_seqlens != nullptr, &pr);
    if (st != KDA_OK) return st;
    int32_t mode, seg_len, debug_flags, sbf;
    int64_t wait_limit;
    if ((st = validate_options(opts, pr, &mode, &seg_len, &wait_limit, &debug_flags, &sbf)) != KDA_OK)
        return st;
    if (pr.T_total > 0 && (!q || !k || !v || !g || !beta || !out))
        return fail(KDA_ERR_INVALID_ARGUMENT, "a required host pointer is NULL");
    if (pr.varlen) {  // host copy of the offsets: check them here
        if (cu_seqlens[0] != 0 || cu_seqlens[pr.N] != pr.T_total)
            return fail(KDA_ERR_INVALID_ARGUMENT, "cu_seqlens must start at 0 and end at T_total");
        for (int n = 0; n < pr.N; ++n)
            if (cu_seqlens[n + 1] < cu_seqlens[n])
                return fail(KDA_ERR_INVALID_ARGUMENT, "cu_seqlens must be non-decreasing");
    }
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    DeviceInfo* di = nullptr;
    if ((st = device_info(dev, &di)) != KDA_OK) return st;
    const size_t se = sbf ? 2 : 4;  // bytes of a state element (the caller's type)
    const Sizes sz = sizes_of(pr, se);
    // Pieces: serial plans only (segment mode needs the whole sequence in one call).
    int32_t plan_mode = mode, plan_len = 0;  // the whole problem's plan, AUTO resolved
    if (mode == KDA_MODE_AUTO) {
        if (pr.varlen) choose_plan_varlen(pr, cu_seqlens, di->resident_clusters, &plan_mode, &plan_len);
        else choose_plan(pr, di->resident_clusters, &plan_mode, &plan_len);
    }
    const int32_t asked = opts ? opts->host_pieces : 0;
    int want = 1;
    if (plan_mode == KDA_MODE_SERIAL)
        want = asked > 0 ? asked
                         : (sz.q + sz.k + sz.v + sz.g + sz.beta >= kHostPipelineMinBytes ? kAutoHostPieces : 1);
    bool blocks = false;
    const std::vector<HostPiece> pieces = host_pieces(pr, cu_seqlens, want, &blocks);
    const int P = (int)pieces.size();
    // A resolved segment plan runs as planned (run() could not see varlen lengths).
    const int32_t piece_mode = (P > 1 || plan_mode == KDA_MODE_SEGMENT) ? plan_mode : mode;
    const int32_t piece_len = (mode == KDA_MODE_AUTO && plan_mode == KDA_MODE_SEGMENT) ? plan_len : seg_len;

    // Device arena: the whole problem's tensors at their natural offsets, the offsets of
    // every piece rebased to its first token, the final states (the caller's type) and,
    // for token blocks, the fp32 state carried from block to block.
    const size_t sb = sz.state;
    const size_t D = kda::kD, st_elems = (size_t)pr.H * D * D;  // one sequence's states
    const size_t cub = pr.varlen ? (size_t)(pr.N + P) * 4 : 0;
    auto up = [](size_t x) { return (x + 255) & ~(size_t)255; };
    const size_t off_q = 0, off_k = off_q + up(sz.q), off_v = off_k + up(sz.k),
                 off_g = off_v + up(sz.v), off_b = off_g + up(sz.g),
                 off_s0 = off_b + up(sz.beta), off_cu = off_s0 + (initial_state ? up(sb) : 0),
                 off_out = off_cu + up(cub), off_fin = off_out + up(sz.out),
                 off_carry = off_fin + (final_state ? up(sb) : 0),
                 total = off_carry + (blocks ? up(st_elems * 4) : 0);
    void* base = nullptr;
    if ((st = get_workspace(dev, stream, kWsHostArena, total, &base)) != KDA_OK) return st;
    HostPipe* hp = nullptr;
    if ((st = get_pipe(dev, stream, &hp)) != KDA_OK) return st;
    char* b = static_cast<char*>(base);
    uint16_t* d_q = reinterpret_cast<uint16_t*>(b + off_q);
    uint16_t* d_k = reinterpret_cast<uint16_t*>(b + off_k);
    uint16_t* d_v = reinterpret_cast<uint16_t*>(b + off_v);
    float* d_g = reinterpret_cast<float*>(b + off_g);
    uint16_t* d_beta = reinterpret_cast<uint16_t*>(b + off_b);
    char* d_s0 = initial_state ? b + off_s0 : nullptr;
    int32_t* d_cu = reinterpret_cast<int32_t*>(b + off_cu);
    uint16_t* d_out = reinterpret_cast<uint16_t*>(b + off_out);
    char* d_fin = final_state ? b + off_fin : nullptr;
    float* d_carry = blocks ? reinterpret_cast<float*>(b + off_carry) : nullptr;
    const char* h_s0 = static_cast<const char*>(initial_state);
    char* h_fin = static_cast<char*>(final_state);
    std::vector<int32_t> cu_rebased;
    std::vector<size_t> cu_at(P, 0);
    if (pr.varlen) {
        cu_rebased.reserve((size_t)pr.N + P);
        for (int i = 0; i < P; ++i) {
            cu_at[i] = cu_rebased.size();
            for (int32_t n = pieces[i].n0; n <= pieces[i].n1; ++n)
                cu_rebased.push_back(cu_seqlens[n] - cu_seqlens[pieces[i].n0]);
        }
    }

    // Every error after the first copy is queued waits for all three streams, so no copy
    // touches the caller's buffers after the call returns.
    auto drain = [&](kda_status s) {
        cudaStreamSynchronize(hp->in);
        cudaStreamSynchronize(hp->out);
        cudaStreamSynchronize(stream);
        return s;
    };
    if ((e = cudaEventRecord(hp->start, stream)) || (e = cudaStreamWaitEvent(hp->in, hp->start, 0)))
        return cuda_fail(e, "copy-in ordering");
    auto h2d = [&](void* dst, const void* src, size_t n) {
        return n ? cudaMemcpyAsync(dst, src, n, cudaMemcpyHostToDevice, hp->in) : cudaSuccess;
    };
    if (pr.varlen && (e = h2d(d_cu, cu_rebased.data(), cu_rebased.size() * 4)))
        return drain(cuda_fail(e, "cudaMemcpyAsync host->device (cu_seqlens)"));
    for (int i = 0; i < P; ++i) {
        const HostPiece& pc = pieces[i];
        const size_t t0 = (size_t)pc.t0, nt = (size_t)(pc.t1 - pc.t0);
        const size_t tq = (size_t)pr.Hq * D, tk = (size_t)pr.Hk * D, tv = (size_t)pr.H * D;
        const size_t s_first = blocks ? 0 : (size_t)pc.n0, s_count = blocks ? (i == 0 ? 1 : 0)
                                                                             : (size_t)(pc.n1 - pc.n0);
        if ((e = h2d(d_q + t0 * tq, q + t0 * tq, nt * tq * 2)) ||
            (e = h2d(d_k + t0 * tk, k + t0 * tk, nt * tk * 2)) ||
            (e = h2d(d_v + t0 * tv, v + t0 * tv, nt * tv * 2)) ||
            (e = h2d(d_g + t0 * tv, g + t0 * tv, nt * tv * 4)) ||
            (e = h2d(d_beta + t0 * pr.H, beta + t0 * pr.H, nt * pr.H * 2)) ||
            (initial_state && (e = h2d(d_s0 + s_first * st_elems * se, h_s0 + s_first * st_elems * se,
                                       s_count * st_elems * se))) ||
            (e = cudaEventRecord(hp->in_done[i], hp->in)))
            return drain(cuda_fail(e, "cudaMemcpyAsync host->device"));
    }
    // Compute every piece on the caller's stream, each after its own copy-in.
    for (int i = 0; i < P; ++i) {
        const HostPiece& pc = pieces[i];
        Problem pp = pr;
        pp.T_total = pc.t1 - pc.t0;
        if (blocks) {
            pp.N = 1;
            pp.varlen = false;
            pp.dense_len = pp.T_total;
        } else {
            pp.N = pc.n1 - pc.n0;
        }
        const size_t t0 = (size_t)pc.t0, n0 = blocks ? 0 : (size_t)pc.n0;
        // Token blocks: the first reads the caller's initial state, later ones the fp32
        // carry; every block but the last writes the carry, the last the final state.
        const void* s0 = nullptr;
        void* sfin = nullptr;
        int32_t s0_bf = sbf, fin_bf = sbf;
        if (blocks) {
            if (i > 0) {
                s0 = d_carry;
                s0_bf = 0;
            } else {
                s0 = d_s0;
            }
            if (i < P - 1) {
                sfin = d_carry;
                fin_bf = 0;
            } else {
                sfin = d_fin;
            }
        } else {
            s0 = d_s0 ? d_s0 + n0 * st_elems * se : nullptr;
            sfin = d_fin ? d_fin + n0 * st_elems * se : nullptr;
        }
        if ((e = cudaStreamWaitEvent(stream, hp->in_done[i], 0)))
            return drain(cuda_fail(e, "cudaStreamWaitEvent"));
        st = run(pp, d_q + t0 * pr.Hq * D, d_k + t0 * pr.Hk * D, d_v + t0 * pr.H * D,
                 d_g + t0 * pr.H * D, d_beta + t0 * pr.H, scale, s0, s0_bf,
                 pr.varlen ? d_cu + cu_at[i] : nullptr, d_out + t0 * pr.Ho * D, sfin, fin_bf, stream,
                 piece_mode, piece_len, wait_limit, debug_flags);
        if (st != KDA_OK) return drain(st);
        if ((e = cudaEventRecord(hp->computed[i], stream)))
            return drain(cuda_fail(e, "cudaEventRecord"));
    }
    // Copy out each piece once it has computed (final states of whole sequences with their
    // piece; a carried state after the last block).
    for (int i = 0; i < P; ++i) {
        const HostPiece& pc = pieces[i];
        const size_t t0 = (size_t)pc.t0, nt = (size_t)(pc.t1 - pc.t0), to = (size_t)pr.Ho * D;
        if ((e = cudaStreamWaitEvent(hp->out, hp->computed[i], 0)))
            return drain(cuda_fail(e, "cudaStreamWaitEvent"));
        if (nt && (e = cudaMemcpyAsync(out + t0 * to, d_out + t0 * to, nt * to * 2,
                                       cudaMemcpyDeviceToHost, hp->out)))
            return drain(cuda_fail(e, "cudaMemcpyAsync device->host (out)"));
        const bool fin_now = final_state && (blocks ? i == P - 1 : pc.n1 > pc.n0);
        const size_t n0 = blocks ? 0 : (size_t)pc.n0, nn = blocks ? 1 : (size_t)(pc.n1 - pc.n0);
        if (fin_now && (e = cudaMemcpyAsync(h_fin + n0 * st_elems * se, d_fin + n0 * st_elems * se,
                                            nn * st_elems * se, cudaMemcpyDeviceToHost, hp->out)))
            return drain(cuda_fail(e, "cudaMemcpyAsync device->host (final_state)"));
    }
    if ((e = cudaEventRecord(hp->out_done, hp->out)) || (e = cudaStreamWaitEvent(stream, hp->out_done, 0)))
        return drain(cuda_fail(e, "copy-out ordering"));
    if ((e = cudaStreamSynchronize(stream))) return drain(cuda_fail(e, "cudaStreamSynchronize"));
    return KDA_OK;
}

kda_status kda_workspace_bytes(const kda_shape* shape, const kda_options* opts, size_t* bytes) {
    t_last_error[0] = '\0';
    if (!bytes) return fail(KDA_ERR_INVALID_ARGUMENT, "bytes is NULL");
    Problem pr{};
    kda_status st = validate_shape(shape, shape && shape->num_seqs > 0, &pr);
    if (st != KDA_OK) return st;
    int32_t mode, seg_len, debug_flags;
    int64_t wait_limit;
    if ((st = validate_options(opts, pr, &mode, &seg_len, &wait_limit, &debug_flags)) != KDA_OK)
        return st;
    if (mode == KDA_MODE_SEGMENT && pr.varlen) {
        *bytes = plan_segments_varlen(pr, seg_len).bytes;
        return KDA_OK;
    }
    if (mode == KDA_MODE_AUTO) {
        int dev = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
        DeviceInfo* di = nullptr;
        if ((st = device_info(dev, &di)) != KDA_OK) return st;
        choose_plan(pr, di->resident_clusters, &mode, &seg_len);
    }
    *bytes = mode == KDA_MODE_SEGMENT ? plan_segments(pr, seg_len).bytes : 0;
    return KDA_OK;
}

kda_status kda_plan(const kda_shape* shape, int32_t varlen, int32_t resident_clusters, int32_t* mode,
                    int32_t* segment_len) {
    t_last_error[0] = '\0';
    if (!mode || !segment_len) return fail(KDA_ERR_INVALID_ARGUMENT, "mode or segment_len is NULL");
    if (resident_clusters < 1) return fail(KDA_ERR_INVALID_ARGUMENT, "resident_clusters must be >= 1");
    Problem pr{};
    kda_status st = validate_shape(shape, varlen != 0, &pr);
    if (st != KDA_OK) return st;
    choose_plan(pr, resident_clusters, mode, segment_len);
    return KDA_OK;
}

kda_status kda_plan_varlen(const kda_shape* shape, const int32_t* host_cu_seqlens, int32_t resident_clusters,
                           int32_t* mode, int32_t* segment_len) {
    t_last_error[0] = '\0';
    if (!mode || !segment_len) return fail(KDA_ERR_INVALID_ARGUMENT, "mode or segment_len is NULL");
    if (resident_clusters < 1) return fail(KDA_ERR_INVALID_ARGUMENT, "resident_clusters must be >= 1");
    if (!host_cu_seqlens) return fail(KDA_ERR_INVALID_ARGUMENT, "host_cu_seqlens is NULL");
    Problem pr{};
    kda_status st = validate_shape(shape, true, &pr);
    if (st != KDA_OK) return st;
    if (host_cu_seqlens[0] != 0 || host_cu_seqlens[pr.N] != pr.T_total)
        return fail(KDA_ERR_INVALID_ARGUMENT, "cu_seqlens must start at 0 and end at T_total");
    for (int n = 0; n < pr.N; ++n)
        if (host_cu_seqlens[n + 1] < host_cu_seqlens[n])
            return fail(KDA_ERR_INVALID_ARGUMENT, "cu_seqlens must be non-decreasing");
    choose_plan_varlen(pr, host_cu_seqlens, resident_clusters, mode, segment_len);
    return KDA_OK;
}

kda_status kda_decode(const kda_shape* shape, const uint16_t* q, const uint16_t* k,
                      const uint16_t* v, const float* g, const uint16_t* beta, float scale,
                      const void* initial_state, void* final_state, int32_t state_dtype,
                      uint16_t* out, void* stream) {
    t_last_error[0] = '\0';
    Problem pr{};
    kda_status st = validate_shape(shape, false, &pr);
    if (st != KDA_OK) return st;
    if (state_dtype != KDA_STATE_F32 && state_dtype != KDA_STATE_BF16)
        return fail(KDA_ERR_INVALID_ARGUMENT, "unknown state_dtype %d", state_dtype);
    const size_t elem = state_dtype == KDA_STATE_BF16 ? 2 : 4;
    if ((st = validate_pointers(pr, q, k, v, g, beta, scale, initial_state, nullptr, out,
                                final_state, elem)) != KDA_OK)
        return st;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    DeviceInfo* di = nullptr;
    if ((st = device_info(dev, &di)) != KDA_OK) return st;
    if (pr.T_total == 0 && !final_state) return KDA_OK;
    kda::DecodeParams p{};
    p.q = reinterpret_cast<const __nv_bfloat16*>(q);
    p.k = reinterpret_cast<const __nv_bfloat16*>(k);
    p.v = reinterpret_cast<const __nv_bfloat16*>(v);
    p.g = g;
    p.beta = reinterpret_cast<const __nv_bfloat16*>(beta);
    p.s0 = initial_state;
    p.sfin = final_state;
    p.out = reinterpret_cast<__nv_bfloat16*>(out);
    p.T = pr.dense_len;
    p.N = pr.N;
    p.H = pr.H;
    p.Hq = pr.Hq;
    p.scale = scale;
    p.state_bf16 = state_dtype == KDA_STATE_BF16;
    if ((e = kda::launch_decode(p, (cudaStream_t)stream)) != cudaSuccess)
        return cuda_fail(e, "decode kernel launch");
    return KDA_OK;
}

kda_status kda_get_device_status(void* stream, int32_t* code) {
    t_last_error[0] = '\0';
    if (!code) return fail(KDA_ERR_INVALID_ARGUMENT, "code is NULL");
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    DeviceInfo* di = nullptr;
    kda_status st = device_info(dev, &di);
    if (st != KDA_OK) return st;
    if ((e = cudaStreamSynchronize((cudaStream_t)stream))) return cuda_fail(e, "cudaStreamSynchronize");
    int32_t host = 0;
    if ((e = cudaMemcpy(&host, di->status, sizeof(host), cudaMemcpyDeviceToHost)))
        return cuda_fail(e, "cudaMemcpy(status word)");
    const int32_t zero = 0;
    if ((e = cudaMemcpy(di->status, &zero, sizeof(zero), cudaMemcpyHostToDevice)))
        return cuda_fail(e, "cudaMemcpy(status word reset)");
    *code = host;
    return KDA_OK;
}

kda_status kda_release_workspaces(int32_t device) {
    t_last_error[0] = '\0';
    std::lock_guard<std::mutex> lock(g_mutex);
    int cur = 0;
    cudaGetDevice(&cur);
    for (size_t i = 0; i < g_workspaces.size();) {
        if (device < 0 || g_workspaces[i].device == device) {
            cudaSetDevice(g_workspaces[i].device);
            cudaDeviceSynchronize();
            cudaFree(g_workspaces[i].ptr);
            g_workspaces.erase(g_workspaces.begin() + i);
        } else {
            ++i;
        }
    }
    for (size_t i = 0; i < g_pipes.size();) {
        if (device < 0 || g_pipes[i]->device == device) {
            destroy_pipe(*g_pipes[i]);
            g_pipes.erase(g_pipes.begin() + i);
        } else {
            ++i;
        }
    }
    cudaSetDevice(cur);
    return KDA_OK;
}

const char* kda_status_string(kda_status s) {
    switch (s) {
        case KDA_OK: return "KDA_OK";
        case KDA_ERR_INVALID_ARGUMENT: return "KDA_ERR_INVALID_ARGUMENT";
        case KDA_ERR_ALIASING: return "KDA_ERR_ALIASING";
        case KDA_ERR_UNSUPPORTED_DEVICE: return "KDA_ERR_UNSUPPORTED_DEVICE";
        case KDA_ERR_OUT_OF_MEMORY: return "KDA_ERR_OUT_OF_MEMORY";
        case KDA_ERR_CUDA: return "KDA_ERR_CUDA";
        case KDA_ERR_CAPTURE_NEEDS_WARMUP: return "KDA_ERR_CAPTURE_NEEDS_WARMUP";
        case KDA_ERR_DEVICE_TIMEOUT: return "KDA_ERR_DEVICE_TIMEOUT";
    }
    return "KDA_ERR_UNKNOWN";
}

const char* kda_last_error_message(void) { return t_last_error; }

const char* kda_version(void) { return "0.1.0"; }

}  // extern "C"

// ---------------------------------------------------------------------------
// Segment-parallel prefill that allocates nothing on the device.
//
// Some callers cannot call cudaMalloc at all: applications whose caching allocator owns
// every byte of device memory and forbids side allocations, real-time services that must
// not risk an allocation failure or the device synchronisation a cudaMalloc can imply in
// the middle of a request, and plugin hosts that give a library no allocation rights.
// kda_prefill_segment_noalloc() serves them: its scratch (segment summaries, transitions
// and carries) lives in one fixed file-scope device array, so no call allocates or frees
// anything.
namespace {

// 32 MiB: room for 512 fp32 128x128 state slots; a call needs B * H * (3 * nseg - 2).
constexpr size_t kNoAllocScratchBytes = (size_t)32 << 20;

struct NoAllocDevice {
    bool ready = false;
    void* scratch = nullptr;
};
NoAllocDevice g_noalloc[kMaxDevices];  // guarded by g_mutex

}  // namespace

// Held by every GPU that loads this library, until the process exits.  Host code must
// not pass this name to a kernel: on the host it is only a stand-in for the symbol.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

namespace {

// Device address of the scratch array on `dev` (the current device), looked up once
// per device with cudaGetSymbolAddress.
kda_status noalloc_scratch(int dev, void** out) {
    std::lock_guard<std::mutex> lock(g_mutex);
    NoAllocDevice& d = g_noalloc[dev];
    if (!d.ready) {
        void* ptr = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
        if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(no-allocation scratch)");
        d.scratch = ptr;
        d.ready = true;
    }
    *out = d.scratch;
    return KDA_OK;
}

}  // namespace

extern "C" kda_status kda_prefill_segment_noalloc(const kda_shape* shape, const uint16_t* q,
                                                  const uint16_t* k, const uint16_t* v,
                                                  const float* g, const uint16_t* beta,
                                                  float scale, const float* initial_state,
                                                  uint16_t* out, float* final_state,
                                                  int32_t segment_len, void* stream_) {
    t_last_error[0] = '\0';
    cudaStream_t stream = (cudaStream_t)stream_;
    Problem pr{};
    kda_status st = validate_shape(shape, false, &pr);
    if (st != KDA_OK) return st;
    if (segment_len <= 0 || segment_len % kda::kChunk != 0)
        return fail(KDA_ERR_INVALID_ARGUMENT,
                    "segment_len must be a positive multiple of 16 (got %d)", segment_len);
    if ((st = validate_pointers(pr, q, k, v, g, beta, scale, initial_state, nullptr, out,
                                final_state)) != KDA_OK)
        return st;
    const SegPlan sp = plan_segments(pr, segment_len);
    if (sp.bytes > kNoAllocScratchBytes)
        return fail(KDA_ERR_INVALID_ARGUMENT,
                    "this shape needs %zu bytes of segment scratch; the no-allocation entry "
                    "point has %zu (at most %zu state slots of 64 KiB, B*H*(3*nseg-2))",
                    sp.bytes, kNoAllocScratchBytes, kNoAllocScratchBytes / (64 * 1024));
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    DeviceInfo* di = nullptr;
    if ((st = device_info(dev, &di)) != KDA_OK) return st;
    void* scratch = nullptr;
    if ((st = noalloc_scratch(dev, &scratch)) != KDA_OK) return st;
    if (pr.T_total == 0 && !final_state) return KDA_OK;

    kda::FwdParams p;
    kda::TensorMaps maps;
    if ((st = prepare_call(pr, q, k, v, g, beta, scale, initial_state, 0, nullptr, out, final_state, 0,
                           kDefaultWaitLimit, 0, di->status, &p, &maps)) != KDA_OK)
        return st;
    if (sp.nseg <= 1) {  // one segment: the plain serial pass, no scratch
        if ((e = kda::launch_serial(p, maps, stream)) != cudaSuccess)
            return cuda_fail(e, "prefill launch");
        return KDA_OK;
    }
    // The same pipeline as segment mode, on the fixed array instead of a workspace.
    return run_dense_segments(pr, p, maps, sp, segment_len, scratch, di->sm_count, stream);
}
