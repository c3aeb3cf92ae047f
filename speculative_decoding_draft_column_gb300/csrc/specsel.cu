// libspecsel: exact per-column top-k and fused greedy verify over bf16 logits
// for one GB300 (sm_103a) -- host side: argument checks, kernel plans,
// scratch, streams and the C ABI.
//
// The operations ("A drafter inside the artifact", Ignis DFlash2 page,
// section "How it works"):
//   * top-k over each draft column of V logits: largest first, ties to the
//     smaller token id (third paragraph);
//   * greedy verify: per target column the argmax (same tie rule), then per
//     lane the longest run of drafts equal to those argmaxes, committed
//     together with the target's own next token (first paragraph).
//
// One kernel launch does a whole round (one streaming pass over the draft and
// target logits; no tensor cores -- the step is a pure reduction bound by HBM
// bandwidth).  Two streaming kernels implement it (round_cta.cuh,
// round_warp.cuh); the host picks by how much each SM streams.

#include <cuda_runtime.h>
#include <stdarg.h>
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include <atomic>
#include <mutex>
#include <string>
#include <vector>

#include "specsel.h"
#include "common.cuh"
#include "round_cta.cuh"
#include "round_warp.cuh"
#include "round_gm.cuh"
#include "head_q4.cuh"

namespace {

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------

constexpr int kMaxDevices = 64;

// Kernel choice.  The CTA-cooperative kernel keeps one threshold per column
// per CTA and wins while an SM streams a few columns at most; the per-warp
// kernel has no coordination inside the stream and wins once every warp sees
// megabytes.  Measured on GB300 (graph-replayed rounds, k = 8 and 20): the
// CTA kernel is ahead up to 6.3 MB of logits per SM (219 against 225 us),
// behind at 26 MB per SM (850 against 696 us); the switch is at 6 MiB.
constexpr int64_t kCtaMaxBytesPerSm = 6ll << 20;
std::atomic<int> g_kernel_choice{SPEC_KERNEL_AUTO};

struct DeviceState {
    bool init = false;
    int sms = 0;
    int occ_w[2][2] = {{0, 0}, {0, 0}};   // per-warp kernel: resident CTAs per SM, [slots-1][mapped]
    int occ_c = 0;                        // CTA kernel: resident CTAs per SM
    int clusters8 = 0;                    // group-maxima one pass in clusters of 8: clusters resident at once
    int col_clusters[9] = {};             // group-maxima whole columns in clusters of Q (2..8): clusters resident at once
    // Scratch: [col tickets and certificates | lane tickets | partial lists].
    // Each region keeps its place and capacity until the whole area is
    // reallocated (and zeroed), so a ticket is never laid over stale data.
    void *scratch = nullptr;
    size_t scratch_bytes = 0;
    int64_t cap_cols = 0, cap_lanes = 0, cap_part = 0;
    // Areas a larger one has replaced.  Launches already enqueued, and CUDA
    // graphs captured earlier, still hold their addresses (and leave their
    // tickets at zero), so they stay allocated until spec_release.
    std::vector<void *> retired;
    void *staging = nullptr;
    size_t staging_bytes = 0;
};

std::mutex g_mu;
DeviceState g_dev[kMaxDevices];
std::atomic<int64_t> g_launches{0};
thread_local cudaStream_t t_stream = nullptr;
thread_local int32_t t_last_kernel = SPEC_KERNEL_AUTO;
thread_local std::string t_err;

spec_status fail(spec_status st, const char *fmt, ...) __attribute__((format(printf, 2, 3)));
spec_status fail(spec_status st, const char *fmt, ...)
{
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    t_err = buf;
    return st;
}

spec_status cuda_fail(cudaError_t e, const char *what)
{
    return fail(SPEC_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorString(e), cudaGetErrorName(e));
}


template <int S, bool M>
void *kernel_ptr() { return reinterpret_cast<void *>(wrp::spec_round_kernel<S, M>); }

spec_status device_state(DeviceState **out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices) return fail(SPEC_ERR_CUDA, "device ordinal %d unsupported", dev);
    DeviceState &d = g_dev[dev];
    if (!d.init) {
        e = cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute");
        void *kw[2][2] = {{kernel_ptr<1, false>(), kernel_ptr<1, true>()},
                          {kernel_ptr<2, false>(), kernel_ptr<2, true>()}};
        for (int s = 0; s < 2; ++s)
            for (int m = 0; m < 2; ++m) {
                e = cudaFuncSetAttribute(kw[s][m], cudaFuncAttributeMaxDynamicSharedMemorySize, (int)wrp::kSmemBytes);
                if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute");
                e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&d.occ_w[s][m], kw[s][m], wrp::kThreads,
                                                                  wrp::kSmemBytes);
                if (e != cudaSuccess) return cuda_fail(e, "cudaOccupancyMaxActiveBlocksPerMultiprocessor");
                if (d.occ_w[s][m] < 1) d.occ_w[s][m] = 1;
            }
        e = cudaFuncSetAttribute(cta::spec_round_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)cta::kSmemBytes);
        if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute");
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&d.occ_c, cta::spec_round_kernel, cta::kThreads,
                                                          cta::kSmemBytes);
        if (e != cudaSuccess) return cuda_fail(e, "cudaOccupancyMaxActiveBlocksPerMultiprocessor");
        if (d.occ_c < 1) d.occ_c = 1;
        {
            // clusters of 8 CTAs of the one-pass kernel that fit on the GPU at once
            e = cudaFuncSetAttribute(reinterpret_cast<void *>(gm::spec_round_kernel<8, 7>),
                                     cudaFuncAttributeMaxDynamicSharedMemorySize, (int)gm::kSmemBytes);
            if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute");
            cudaLaunchConfig_t cfg;
            memset(&cfg, 0, sizeof cfg);
            cfg.gridDim = dim3(8 * 19);
            cfg.blockDim = dim3(gm::kThreads);
            cfg.dynamicSmemBytes = gm::kSmemBytes;
            cudaLaunchAttribute at[1];
            at[0].id = cudaLaunchAttributeClusterDimension;
            at[0].val.clusterDim.x = 8;
            at[0].val.clusterDim.y = 1;
            at[0].val.clusterDim.z = 1;
            cfg.attrs = at;
            cfg.numAttrs = 1;
            int n = 0;
            if (cudaOccupancyMaxActiveClusters(&n, reinterpret_cast<void *>(gm::spec_round_kernel<8, 7>), &cfg) !=
                cudaSuccess) {
                cudaGetLastError();
                n = 0;   // no clusters: the one-pass mode runs without them
            }
            d.clusters8 = n;
            // whole columns in clusters of Q CTAs, Q = 2 .. 8
            void *k8 = reinterpret_cast<void *>(gm::spec_round_kernel<8, 8>);
            e = cudaFuncSetAttribute(k8, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)gm::kSmemInboxBytes);
            if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute");
            for (int q = 2; q <= 8; ++q) {
                cfg.gridDim = dim3((unsigned)(q * (d.sms / q)));
                cfg.dynamicSmemBytes = gm::kSmemInboxBytes;
                at[0].val.clusterDim.x = (unsigned)q;
                int m = 0;
                if (cudaOccupancyMaxActiveClusters(&m, k8, &cfg) != cudaSuccess) {
                    cudaGetLastError();
                    m = 0;
                }
                d.col_clusters[q] = m;
            }
        }
        void *kg[9] = {reinterpret_cast<void *>(gm::spec_round_kernel<8, 3>),
                       reinterpret_cast<void *>(gm::spec_round_kernel<8, 4>),
                       reinterpret_cast<void *>(gm::spec_round_kernel<16, 4>),
                       reinterpret_cast<void *>(gm::spec_round_kernel<1, 0>),
                       reinterpret_cast<void *>(gm::spec_round_kernel<2, 0>),
                       reinterpret_cast<void *>(gm::spec_round_kernel<4, 0>),
                       reinterpret_cast<void *>(gm::spec_round_kernel<8, 0>),
                       reinterpret_cast<void *>(gm::spec_round_kernel<8, 1>),
                       reinterpret_cast<void *>(gm::spec_round_kernel<8, 2>)};
        for (void *k : kg) {
            e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)gm::kSmemBytes);
            if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute");
        }
        d.init = true;
    }
    *out = &d;
    return SPEC_OK;
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

struct ScratchPtrs {
    unsigned int *col_ticket;
    unsigned int *lane_ticket;
    unsigned long long *partials;
};

struct ScratchCaps {
    int64_t cols, lanes, part;   // cols = ticket/certificate words; part = partial-list entries (u64)
};

size_t scratch_bytes(const ScratchCaps &c)
{
    return align256((size_t)c.cols * 4) + align256((size_t)c.lanes * 4) + align256((size_t)c.part * 8);
}

ScratchPtrs scratch_ptrs(const DeviceState &d)
{
    char *p = static_cast<char *>(d.scratch);
    ScratchPtrs s;
    s.col_ticket = reinterpret_cast<unsigned int *>(p);
    p += align256((size_t)d.cap_cols * 4);
    s.lane_ticket = reinterpret_cast<unsigned int *>(p);
    p += align256((size_t)d.cap_lanes * 4);
    s.partials = reinterpret_cast<unsigned long long *>(p);
    return s;
}

bool stream_capturing(cudaStream_t st)
{
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(st, &cs) != cudaSuccess) return false;
    return cs != cudaStreamCaptureStatusNone;
}

// Grow (never shrink) the device's scratch so that every region covers
// `need`; fresh scratch is zeroed, and the kernels leave every ticket at zero
// when they finish.  The area it replaces is retired, not freed.
spec_status ensure_scratch(DeviceState &d, const ScratchCaps &need, cudaStream_t st)
{
    if (d.scratch && need.cols <= d.cap_cols && need.lanes <= d.cap_lanes && need.part <= d.cap_part)
        return SPEC_OK;
    if (stream_capturing(st))
        return fail(SPEC_ERR_ALLOC, "scratch must grow during stream capture; call spec_reserve before capturing");
    auto grow = [](int64_t have, int64_t want) { return want <= have ? have : want + want / 4 + 64; };
    ScratchCaps c;
    c.cols = grow(d.cap_cols, need.cols);
    c.lanes = grow(d.cap_lanes, need.lanes);
    c.part = grow(d.cap_part, need.part);
    const size_t bytes = scratch_bytes(c);
    void *fresh = nullptr;
    cudaError_t e = cudaMalloc(&fresh, bytes);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return fail(SPEC_ERR_ALLOC, "cudaMalloc(%zu) for scratch: %s", bytes, cudaGetErrorString(e));
    }
    e = cudaMemset(fresh, 0, bytes);   // synchronous: zero before any launch can see it
    if (e != cudaSuccess) {
        cudaFree(fresh);
        return cuda_fail(e, "cudaMemset scratch");
    }
    if (d.scratch) d.retired.push_back(d.scratch);
    d.scratch = fresh;
    d.scratch_bytes = bytes;
    d.cap_cols = c.cols;
    d.cap_lanes = c.lanes;
    d.cap_part = c.part;
    return SPEC_OK;
}

int64_t vectors_of(const void *buf, int64_t n_elems)
{
    const int64_t mis = (int64_t)((reinterpret_cast<uintptr_t>(buf) >> 1) & 7);
    return (n_elems + mis + 7) >> 3;
}

// Split the streaming units (warps or CTAs) of a full-GPU grid between the
// draft and the target logits in proportion to their 16-byte vectors, so
// that every unit streams the same number of bytes.  No slice is made
// smaller than min_slice vectors, and the published lists (two per unit,
// kk_stride entries each) must fit in max_partials entries.
void split_units(int64_t nv_d, int64_t nv_t, int64_t max_units, int64_t min_slice, int kk_stride,
                 int64_t max_partials, int32_t *w_d, int32_t *w_t)
{
    int64_t total = max_units;
    const int64_t cap = max_partials / (2 * (int64_t)kk_stride);
    if (total > cap) total = cap;
    if (total < 2) total = 2;
    auto limit = [min_slice](int64_t nv) { const int64_t m = nv / min_slice; return m < 1 ? (int64_t)1 : m; };
    int64_t d = 0, t = 0;
    if (nv_d > 0 && nv_t > 0) {
        d = (int64_t)((double)total * (double)nv_d / (double)(nv_d + nv_t) + 0.5);
        if (d < 1) d = 1;
        if (d > total - 1) d = total - 1;
        t = total - d;
    } else if (nv_d > 0) {
        d = total;
    } else {
        t = total;
    }
    if (nv_d > 0 && d > limit(nv_d)) d = limit(nv_d);
    if (nv_t > 0 && t > limit(nv_t)) t = limit(nv_t);
    *w_d = (int32_t)d;
    *w_t = (int32_t)t;
}

// Which kernel runs a round, and on how many units (filled into a.d_units,
// a.t_units; a.pstride is set too).
struct Plan {
    bool per_cta;
    bool gm;          // the group-maxima kernel
    int gm_u;         // its batch width: 16-byte vectors per thread per batch (1, 2, 4 or 8; one pass: 8 or 16)
    int gm_mode;      // its mode: 0 slices, 1 whole columns per CTA, 2 / 3 whole columns with finishing warps,
                      // 4 one pass (gm_u: loads per thread), 7 one pass in clusters of 8 CTAs a column,
                      // 8 whole columns in clusters of `cluster` CTAs
    int slots;        // per-warp kernel: 2 for k > 32 (finer seed groups)
    bool mapped;
    int64_t grid;     // CTAs
    int64_t partials; // entries (u64) of the partials area the launch uses
    int cluster = 0;  // CTAs a thread-block cluster (the cluster modes; 0: none)
};

// The group-maxima kernel's plan: its mode and the CTAs of each run.  In
// order: one pass in clusters of 8 CTAs a column; one pass (8 or 16 loads a
// thread); whole columns in clusters of 2 to 8 CTAs; whole columns per CTA
// (with finishing warps from 1.5 columns per SM on); and, if slices is set,
// slice mode.  In slice mode every batch must
// touch two columns at most (V >= 8 * 512 * U); of the widths that allow it,
// the widest unless a narrower one cuts the vectors of the most loaded CTA
// by a third: a narrower batch balances small rounds better but gives a
// column's finishing CTA more group keys to read.  False if no mode fits, or
// the scratch it needs would not fit in max_partials entries.
bool plan_gm(const DeviceState &d, RoundArgs &a, int64_t nv_d, int64_t nv_t, int64_t max_partials, bool slices,
             Plan &p)
{
    int64_t vmin = INT64_MAX;
    if (nv_d > 0) vmin = a.d_V < vmin ? a.d_V : vmin;
    if (nv_t > 0) vmin = a.t_V < vmin ? a.t_V : vmin;
    // One pass: the CTAs of each run dealt out to its columns (every column
    // at least one, every CTA at least one vector), every CTA's slice at
    // most 512 L vectors (L = 8 loads per thread, else 16) so that it holds
    // the slice in registers, and a column's published entries (2 kk a CTA)
    // fitting the merge buffer.
    const int kmax = a.k > a.t_k ? a.k : a.t_k;
    // One pass in clusters: eight CTAs a column, each column one cluster,
    // when that keeps at least three quarters of the SMs busy, every
    // cluster is resident at once, and a column's eighth fits 4,096 vectors.
    {
        constexpr int Q = 8;
        const int64_t cols = (nv_d > 0 ? a.d_cols : 0) + (nv_t > 0 ? a.t_cols : 0);
        const int64_t units = Q * cols;
        const int stride = 2 * kmax + 2;
        auto fits8 = [](int64_t nv, int64_t V) { return nv == 0 || ((V / 8 + 2 + Q - 1) / Q <= 512 * 8 && V / 8 >= Q); };
        if (cols > 0 && cols <= d.clusters8 && units <= d.sms && 4 * units >= 3 * (int64_t)d.sms &&
            fits8(nv_d, a.d_V) && fits8(nv_t, a.t_V) && units * stride <= max_partials) {
            a.pstride = stride;
            a.d_units = (int32_t)(nv_d > 0 ? Q * a.d_cols : 0);
            a.t_units = (int32_t)(nv_t > 0 ? Q * a.t_cols : 0);
            p.gm = true;
            p.gm_u = 8;
            p.gm_mode = 7;
            p.grid = units;
            p.partials = units * stride;
            return true;
        }
    }
    for (int L : {8, 16}) {
        const int stride = 2 * kmax + 2;
        int32_t wd = 0, wt = 0;
        split_units(nv_d, nv_t, d.sms, 512, stride, max_partials, &wd, &wt);   // 8 KB a CTA at least
        auto fits = [L](int64_t nv, int64_t cols, int64_t w, int64_t V, int kk) {
            if (nv == 0) return true;
            if (w < cols) return false;
            const int64_t nmin = w / cols, nmax = (w + cols - 1) / cols;
            const int64_t nvc = V / 8 + 2;   // a column's vectors, at most
            return (nvc + nmin - 1) / nmin <= 512 * (int64_t)L && V / 8 >= nmax &&
                   nmax * 2 * kk <= (int64_t)gm::kCap;
        };
        const int64_t units = (nv_d > 0 ? wd : 0) + (nv_t > 0 ? wt : 0);
        if (!fits(nv_d, a.d_cols, wd, a.d_V, a.k) || !fits(nv_t, a.t_cols, wt, a.t_V, a.t_k) ||
            units * stride > max_partials)
            continue;
        a.pstride = stride;
        a.d_units = nv_d > 0 ? wd : 0;
        a.t_units = nv_t > 0 ? wt : 0;
        p.gm = true;
        p.gm_u = L;
        p.gm_mode = 4;
        p.grid = units;
        p.partials = units * a.pstride;
        return true;
    }
    if (vmin < gm::kMinV) return false;
    // Whole columns in clusters: fewer columns than three quarters of the
    // SMs, each column one cluster of Q CTAs (the fewest that keep three
    // quarters of the SMs busy, at most 8), every CTA at least one batch of
    // U = 8 and at most the kKeyRows whose keys it keeps in shared memory,
    // every cluster resident at once.
    {
        int64_t vmax2 = 0;
        if (nv_d > 0) vmax2 = a.d_V > vmax2 ? a.d_V : vmax2;
        if (nv_t > 0) vmax2 = a.t_V > vmax2 ? a.t_V : vmax2;
        const int64_t cols = (nv_d > 0 ? a.d_cols : 0) + (nv_t > 0 ? a.t_cols : 0);
        const int64_t B = 512 * 8;
        for (int Q = 2; Q <= 8 && cols > 0 && vmin >= 8 * B; ++Q) {
            const int64_t units = Q * cols;
            if (units > d.sms) break;
            if (4 * units < 3 * (int64_t)d.sms) continue;
            const int64_t nb_min = (vmin / 8) / B, nb_max = (vmax2 / 8 + 2 + B - 1) / B;
            if (nb_min < Q || (nb_max + Q - 1) / Q > gm::kKeyRows || cols > d.col_clusters[Q]) break;
            a.d_units = (int32_t)(nv_d > 0 ? Q * a.d_cols : 0);
            a.t_units = (int32_t)(nv_t > 0 ? Q * a.t_cols : 0);
            p.gm = true;
            p.gm_u = 8;
            p.gm_mode = 8;
            p.cluster = Q;
            p.grid = units;
            p.partials = 0;
            return true;
        }
    }
    // Column mode: at least three quarters as many columns as SMs, every
    // column at least one batch of U = 8 and at most the kKeyRows batches
    // whose keys a CTA keeps in shared memory.  Each CTA then owns whole
    // columns: no tickets, no keys in global memory.
    const int64_t cols_all = (nv_d > 0 ? a.d_cols : 0) + (nv_t > 0 ? a.t_cols : 0);
    int64_t vmax = 0;
    if (nv_d > 0) vmax = a.d_V > vmax ? a.d_V : vmax;
    if (nv_t > 0) vmax = a.t_V > vmax ? a.t_V : vmax;
    // With at least 1.5 columns per SM, finishing warps take the columns'
    // finish off the stream: 4 of the 16 warps, or 8 where a column's finish
    // outweighs its stream (k above 8 on columns of at most 192 K logits:
    // GB300, C5s at k = 20 / 64: 196 / 288 us with 4, 177 / 197 with 8; C4
    // and C5 at k = 8 faster with 4).  Columns must fit kTeamRows batches.
    const bool eight = kmax > 8 && vmax <= 192 * 1024 &&
                       (vmax / 8 + 2) <= (int64_t)gm::Team<8>::kTeamRows * gm::Team<8>::kStreamThreads * 8;
    const bool four = (vmax / 8 + 2) <= (int64_t)gm::Team<12>::kTeamRows * gm::Team<12>::kStreamThreads * 8;
    const bool team = 2 * cols_all >= 3 * (int64_t)d.sms && (eight || four);
    if (4 * cols_all >= 3 * (int64_t)d.sms && vmin >= 8 * 512 * 8 && (vmax / 8 + 2) <= (int64_t)gm::kKeyRows * 512 * 8) {
        const int64_t W = cols_all < d.sms ? cols_all : d.sms;
        int64_t ud = 0, ut = 0;
        if (nv_d > 0 && nv_t > 0) {
            ud = (W * a.d_cols + cols_all / 2) / cols_all;
            if (ud < 1) ud = 1;
            if (ud > W - 1) ud = W - 1;
            if (ud > a.d_cols) ud = a.d_cols;
            ut = W - ud < a.t_cols ? W - ud : a.t_cols;
        } else if (nv_d > 0) {
            ud = W;
        } else {
            ut = W;
        }
        a.d_units = (int32_t)ud;
        a.t_units = (int32_t)ut;
        p.gm = true;
        p.gm_u = 8;
        p.gm_mode = !team ? 1 : eight ? 3 : 2;
        p.grid = ud + ut;
        p.partials = 0;
        return true;
    }
    if (!slices) return false;
    int32_t wd = 0, wt = 0;
    split_units(nv_d, nv_t, d.sms, 512, 1, INT64_MAX / 4, &wd, &wt);
    auto nbatches = [](int64_t nv, int64_t B) { return (nv + B - 1) / B; };
    auto most = [&](int64_t nv, int64_t w, int64_t B) -> int64_t {
        if (nv == 0) return 0;
        const int64_t nb = nbatches(nv, B), ww = w < nb ? w : nb;
        return (nb + ww - 1) / ww * B;
    };
    int best = 0;
    int64_t best_cost = 0;
    for (int u : {8, 4, 2, 1}) {
        const int64_t B = 512 * (int64_t)u;
        if (8 * B > vmin) continue;
        const int64_t cd = most(nv_d, wd, B), ct = most(nv_t, wt, B);
        const int64_t c = cd > ct ? cd : ct;
        if (best == 0 || c * 3 < best_cost * 2) {
            best = u;
            best_cost = c;
        }
    }
    if (best == 0) return false;
    const int64_t B = 512 * (int64_t)best;
    const int64_t nbd = nbatches(nv_d, B), nbt = nbatches(nv_t, B);
    const int64_t bytes = (nbd + nbt + a.d_cols + a.t_cols) * 512 * 2;
    const int64_t entries = (bytes + 7) / 8;
    if (entries > max_partials) return false;
    a.d_units = (int32_t)(nv_d > 0 ? (wd < nbd ? wd : nbd) : 0);
    a.t_units = (int32_t)(nv_t > 0 ? (wt < nbt ? wt : nbt) : 0);
    p.gm = true;
    p.gm_u = best;
    p.gm_mode = 0;
    p.grid = (int64_t)a.d_units + a.t_units;
    p.partials = entries;
    return true;
}

// gm_max: the most partials entries the group-maxima kernel may use (the
// area's present size while a graph is being captured); without room, or
// with columns too short for it, the CTA kernel runs instead.
Plan plan_round(const DeviceState &d, RoundArgs &a, int64_t nv_d, int64_t nv_t, bool mapped, int64_t max_partials,
                int64_t gm_max = INT64_MAX)
{
    Plan p;
    const int choice = g_kernel_choice.load(std::memory_order_relaxed);
    const bool small = (nv_d + nv_t) * 16 <= kCtaMaxBytesPerSm * (int64_t)d.sms;
    p.gm = false;
    p.gm_u = 0;
    p.gm_mode = 0;
    p.mapped = mapped;
    const int kmax = a.k > a.t_k ? a.k : a.t_k;   // the larger list of the two runs
    p.slots = kmax > 32 ? 2 : 1;
    a.pstride = kmax + 2;
    // The group-maxima kernel: its column modes at any size, its slice mode
    // up to 6 MiB of logits per SM (its group keys live in scratch).
    if ((choice == SPEC_KERNEL_GROUPMAX || choice == SPEC_KERNEL_AUTO) &&
        plan_gm(d, a, nv_d, nv_t, max_partials < gm_max ? max_partials : gm_max,
                choice == SPEC_KERNEL_GROUPMAX || small, p))
        return p;
    p.per_cta = choice == SPEC_KERNEL_CTA || choice == SPEC_KERNEL_GROUPMAX || (choice == SPEC_KERNEL_AUTO && small);
    if (p.per_cta) {
        split_units(nv_d, nv_t, (int64_t)d.sms * d.occ_c, cta::kMinSliceVec, a.pstride, max_partials, &a.d_units,
                    &a.t_units);
        p.grid = (int64_t)a.d_units + a.t_units;
    } else {
        const int64_t max_warps = (int64_t)d.sms * d.occ_w[p.slots - 1][mapped ? 1 : 0] * wrp::kWarpsPerCta;
        split_units(nv_d, nv_t, max_warps, wrp::kMinSliceVec, a.pstride, max_partials, &a.d_units, &a.t_units);
        p.grid = ((int64_t)a.d_units + a.t_units + wrp::kWarpsPerCta - 1) / wrp::kWarpsPerCta;
    }
    p.partials = ((int64_t)a.d_units + a.t_units) * 2 * a.pstride;   // two lists per unit
    return p;
}

// Launch, with programmatic stream serialization when pdl: the kernel
// signals its dependents at entry and waits for its predecessor before any
// memory access, so the stream order holds while the next launch's setup
// overlaps the current launch's tail.
template <typename K>
cudaError_t launch_pdl(K kernel, unsigned grid, unsigned block, size_t smem, cudaStream_t stream, const RoundArgs &a,
                       bool pdl, unsigned cluster = 0)
{
    cudaLaunchConfig_t cfg;
    memset(&cfg, 0, sizeof cfg);
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(block);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    unsigned na = 0;
    if (pdl) {
        attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[na].val.programmaticStreamSerializationAllowed = 1;
        ++na;
    }
    if (cluster) {
        attr[na].id = cudaLaunchAttributeClusterDimension;
        attr[na].val.clusterDim.x = cluster;
        attr[na].val.clusterDim.y = 1;
        attr[na].val.clusterDim.z = 1;
        ++na;
    }
    cfg.attrs = attr;
    cfg.numAttrs = na;
    return cudaLaunchKernelEx(&cfg, kernel, a);
}

// pdl: whether a CTA-kernel launch may overlap the stream's previous kernel
// (off when a non-kernel operation the kernel depends on comes right before
// it).  Only the CTA kernel -- small, launch-bound rounds -- uses it; it
// measured slower for the per-warp kernel's large rounds.
cudaError_t launch_plan(const Plan &p, const RoundArgs &a, cudaStream_t stream, bool pdl = true)
{
    const unsigned g = (unsigned)p.grid;
    if (p.gm) {
        const size_t m = gm::kSmemBytes;
        if (p.gm_mode == 7) return launch_pdl(gm::spec_round_kernel<8, 7>, g, gm::kThreads, m, stream, a, pdl, 8);
        if (p.gm_mode == 8)
            return launch_pdl(gm::spec_round_kernel<8, 8>, g, gm::kThreads, gm::kSmemInboxBytes, stream, a, pdl,
                              (unsigned)p.cluster);
        if (p.gm_mode == 4 && p.gm_u == 16)
            return launch_pdl(gm::spec_round_kernel<16, 4>, g, gm::kThreads, m, stream, a, pdl);
        if (p.gm_mode == 4) return launch_pdl(gm::spec_round_kernel<8, 4>, g, gm::kThreads, m, stream, a, pdl);
        if (p.gm_mode == 3) return launch_pdl(gm::spec_round_kernel<8, 3>, g, gm::kThreads, m, stream, a, pdl);
        if (p.gm_mode == 2) return launch_pdl(gm::spec_round_kernel<8, 2>, g, gm::kThreads, m, stream, a, pdl);
        if (p.gm_mode == 1) return launch_pdl(gm::spec_round_kernel<8, 1>, g, gm::kThreads, m, stream, a, pdl);
        switch (p.gm_u) {
        case 8: return launch_pdl(gm::spec_round_kernel<8, 0>, g, gm::kThreads, m, stream, a, pdl);
        case 4: return launch_pdl(gm::spec_round_kernel<4, 0>, g, gm::kThreads, m, stream, a, pdl);
        case 2: return launch_pdl(gm::spec_round_kernel<2, 0>, g, gm::kThreads, m, stream, a, pdl);
        default: return launch_pdl(gm::spec_round_kernel<1, 0>, g, gm::kThreads, m, stream, a, pdl);
        }
    }
    if (p.per_cta) return launch_pdl(cta::spec_round_kernel, g, cta::kThreads, cta::kSmemBytes, stream, a, pdl);
    const unsigned b = wrp::kThreads;
    const size_t m = wrp::kSmemBytes;
    if (p.slots == 1 && !p.mapped) return launch_pdl(wrp::spec_round_kernel<1, false>, g, b, m, stream, a, false);
    if (p.slots == 1) return launch_pdl(wrp::spec_round_kernel<1, true>, g, b, m, stream, a, false);
    if (!p.mapped) return launch_pdl(wrp::spec_round_kernel<2, false>, g, b, m, stream, a, false);
    return launch_pdl(wrp::spec_round_kernel<2, true>, g, b, m, stream, a, false);
}

int32_t plan_kernel(const Plan &p) { return p.gm ? SPEC_KERNEL_GROUPMAX : p.per_cta ? SPEC_KERNEL_CTA : SPEC_KERNEL_WARP; }

bool misaligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) != 0; }

spec_status check_topk_args(const uint16_t *logits, int64_t cols, int64_t V, int32_t k, const void *vals,
                            const void *ids)
{
    if (cols < 0) return fail(SPEC_ERR_ARG, "cols = %lld < 0", (long long)cols);
    if (V < 1 || V > INT32_MAX) return fail(SPEC_ERR_ARG, "V = %lld outside [1, 2^31-1]", (long long)V);
    if (k < 1 || k > SPEC_MAX_K || (int64_t)k > V)
        return fail(SPEC_ERR_ARG, "k = %d outside [1, min(V, %d)]", k, SPEC_MAX_K);
    if (cols == 0) return SPEC_OK;
    if (!logits || !vals || !ids) return fail(SPEC_ERR_ARG, "null pointer");
    if (misaligned(logits, 2) || misaligned(vals, 2) || misaligned(ids, 4))
        return fail(SPEC_ERR_ARG, "misaligned pointer (logits/out_vals need 2 bytes, out_ids 4)");
    if (cols > INT64_MAX / V) return fail(SPEC_ERR_ARG, "cols * V overflows");
    return SPEC_OK;
}

spec_status check_verify_args(const uint16_t *tl, const int32_t *drafts, int64_t lanes, int32_t gamma,
                              int64_t V, const int32_t *acc, const int32_t *com)
{
    if (lanes < 0) return fail(SPEC_ERR_ARG, "lanes = %lld < 0", (long long)lanes);
    if (gamma < 1 || gamma > SPEC_MAX_GAMMA)
        return fail(SPEC_ERR_ARG, "gamma = %d outside [1, %d]", gamma, SPEC_MAX_GAMMA);
    if (V < 1 || V > INT32_MAX) return fail(SPEC_ERR_ARG, "V = %lld outside [1, 2^31-1]", (long long)V);
    if (lanes == 0) return SPEC_OK;
    if (!tl || !drafts || !acc || !com) return fail(SPEC_ERR_ARG, "null pointer");
    if (misaligned(tl, 2) || misaligned(drafts, 4) || misaligned(acc, 4) || misaligned(com, 4))
        return fail(SPEC_ERR_ARG, "misaligned pointer");
    if (lanes > INT64_MAX / ((int64_t)(gamma + 1) * V)) return fail(SPEC_ERR_ARG, "lanes * (gamma+1) * V overflows");
    return SPEC_OK;
}

// Plan and launch one kernel covering a top-k part and/or a verify part.
// Sampled verify parameters (uniforms == nullptr: greedy verify).
struct Sampling {
    int32_t top_k = 1;
    double temperature = 1.0, top_p = 1.0;
    const double *uniforms = nullptr;
};

// The caller holds g_mu.
spec_status launch_round_locked(const uint16_t *draft, int64_t cols, int64_t V, int32_t k, const int32_t *id_map,
                                uint16_t *vals, int32_t *ids, const uint16_t *target, const int32_t *drafts,
                                int64_t lanes, int32_t gamma, int64_t tV, int32_t *acc, int32_t *com,
                                spec_counters *counters = nullptr, const Sampling &smp = Sampling())
{
    if (cols == 0 && lanes == 0) return SPEC_OK;
    DeviceState *d = nullptr;
    spec_status st = device_state(&d);
    if (st != SPEC_OK) return st;
    const bool mapped = cols > 0 && id_map != nullptr;
    const int64_t t_cols = lanes * (gamma + 1);

    RoundArgs a;
    memset(&a, 0, sizeof a);
    a.draft = draft; a.d_cols = cols; a.d_V = cols ? V : 1; a.k = cols ? k : 1;
    a.id_map = id_map; a.out_vals = vals; a.out_ids = ids;
    a.target = target; a.t_cols = t_cols; a.t_V = lanes ? tV : 1; a.gamma = gamma;
    a.drafts = drafts; a.out_accept = acc; a.out_commit = com;
    a.counters = lanes ? counters : nullptr;
    a.t_k = lanes && smp.uniforms ? smp.top_k : 1;
    a.temperature = smp.temperature;
    a.top_p = smp.top_p;
    a.uniforms = lanes ? smp.uniforms : nullptr;
    cudaStream_t stream = t_stream;
    const Plan plan = plan_round(*d, a, cols ? vectors_of(draft, cols * V) : 0,
                                 lanes ? vectors_of(target, t_cols * tV) : 0, mapped, INT64_MAX / 4,
                                 stream_capturing(stream) ? d->cap_part : INT64_MAX);
    const ScratchCaps need = {2 * (cols + t_cols), lanes, plan.partials};
    st = ensure_scratch(*d, need, stream);
    if (st != SPEC_OK) return st;
    const ScratchPtrs sp = scratch_ptrs(*d);
    a.partials = sp.partials;
    a.gkeys = reinterpret_cast<uint16_t *>(sp.partials);
    a.col_ticket = sp.col_ticket;
    a.col_cert = sp.col_ticket + (cols + t_cols);
    a.lane_ticket = sp.lane_ticket;
    const cudaError_t e = launch_plan(plan, a, stream);
    if (e != cudaSuccess) return cuda_fail(e, "kernel launch");
    g_launches.fetch_add(1, std::memory_order_relaxed);
    t_last_kernel = plan_kernel(plan);
    return SPEC_OK;
}

spec_status launch_round(const uint16_t *draft, int64_t cols, int64_t V, int32_t k, const int32_t *id_map,
                         uint16_t *vals, int32_t *ids, const uint16_t *target, const int32_t *drafts,
                         int64_t lanes, int32_t gamma, int64_t tV, int32_t *acc, int32_t *com,
                         spec_counters *counters = nullptr, const Sampling &smp = Sampling())
{
    if (cols == 0 && lanes == 0) return SPEC_OK;
    std::lock_guard<std::mutex> lock(g_mu);
    return launch_round_locked(draft, cols, V, k, id_map, vals, ids, target, drafts, lanes, gamma, tV, acc, com,
                               counters, smp);
}

// Grow the host-call staging area; the caller holds g_mu.  The area it
// replaces is retired (freed by spec_release), never freed under a copy
// that may still be in flight.
spec_status ensure_staging(DeviceState &d, size_t bytes)
{
    if (d.staging_bytes >= bytes) return SPEC_OK;
    void *fresh = nullptr;
    const cudaError_t e = cudaMalloc(&fresh, bytes);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return fail(SPEC_ERR_ALLOC, "cudaMalloc(%zu) for staging: %s", bytes, cudaGetErrorString(e));
    }
    if (d.staging) d.retired.push_back(d.staging);
    d.staging = fresh;
    d.staging_bytes = bytes;
    return SPEC_OK;
}

}  // namespace

// ---------------------------------------------------------------------------
// C ABI
// ---------------------------------------------------------------------------

extern "C" {

spec_status spec_topk(const uint16_t *logits, int64_t cols, int64_t V, int32_t k, uint16_t *out_vals,
                      int32_t *out_ids)
{
    t_err.clear();
    spec_status st = check_topk_args(logits, cols, V, k, out_vals, out_ids);
    if (st != SPEC_OK) return st;
    return launch_round(logits, cols, V, k, nullptr, out_vals, out_ids, nullptr, nullptr, 0, 1, 1, nullptr,
                        nullptr);
}

spec_status spec_topk_mapped(const uint16_t *logits, int64_t cols, int64_t V, int32_t k, const int32_t *id_map,
                             uint16_t *out_vals, int32_t *out_ids)
{
    t_err.clear();
    spec_status st = check_topk_args(logits, cols, V, k, out_vals, out_ids);
    if (st != SPEC_OK) return st;
    if (cols > 0 && (!id_map || misaligned(id_map, 4))) return fail(SPEC_ERR_ARG, "id_map null or misaligned");
    return launch_round(logits, cols, V, k, cols > 0 ? id_map : nullptr, out_vals, out_ids, nullptr, nullptr, 0,
                        1, 1, nullptr, nullptr);
}

spec_status spec_verify_v(const uint16_t *target_logits, const int32_t *drafts, int64_t lanes, int32_t gamma,
                          int64_t V, int32_t *out_accept_len, int32_t *out_commit_ids)
{
    t_err.clear();
    spec_status st = check_verify_args(target_logits, drafts, lanes, gamma, V, out_accept_len, out_commit_ids);
    if (st != SPEC_OK) return st;
    return launch_round(nullptr, 0, 1, 1, nullptr, nullptr, nullptr, target_logits, drafts, lanes, gamma, V,
                        out_accept_len, out_commit_ids);
}

spec_status check_sampling(double temperature, double top_p, int32_t top_k, int64_t V, int64_t lanes,
                           const double *uniforms)
{
    if (!(temperature > 0.0) || temperature > 1e30)
        return fail(SPEC_ERR_ARG, "temperature = %g: must be positive and finite", temperature);
    if (!(top_p > 0.0 && top_p <= 1.0)) return fail(SPEC_ERR_ARG, "top_p = %g outside (0, 1]", top_p);
    if (top_k < 1 || top_k > SPEC_MAX_K || (int64_t)top_k > V)
        return fail(SPEC_ERR_ARG, "top_k = %d outside [1, min(V, %d)]", top_k, SPEC_MAX_K);
    if (lanes > 0 && (!uniforms || misaligned(uniforms, 8))) return fail(SPEC_ERR_ARG, "uniforms null or misaligned");
    return SPEC_OK;
}

spec_status spec_round_sampled(const uint16_t *draft_logits, int64_t cols, int64_t V, int32_t k, uint16_t *out_vals,
                               int32_t *out_ids, const uint16_t *target_logits, const int32_t *drafts, int64_t lanes,
                               int32_t gamma, double temperature, double top_p, int32_t top_k,
                               const double *uniforms, int32_t *out_accept_len, int32_t *out_commit_ids)
{
    t_err.clear();
    spec_status st = check_topk_args(draft_logits, cols, V, k, out_vals, out_ids);
    if (st != SPEC_OK) return st;
    st = check_verify_args(target_logits, drafts, lanes, gamma, V, out_accept_len, out_commit_ids);
    if (st != SPEC_OK) return st;
    st = check_sampling(temperature, top_p, top_k, V, lanes, uniforms);
    if (st != SPEC_OK) return st;
    Sampling smp;
    smp.top_k = top_k;
    smp.temperature = temperature;
    smp.top_p = top_p;
    smp.uniforms = uniforms;
    return launch_round(draft_logits, cols, V, k, nullptr, out_vals, out_ids, target_logits, drafts, lanes, gamma,
                        V, out_accept_len, out_commit_ids, nullptr, smp);
}

spec_status spec_verify_sampled(const uint16_t *target_logits, const int32_t *drafts, int64_t lanes, int32_t gamma,
                                int64_t V, double temperature, double top_p, int32_t top_k, const double *uniforms,
                                int32_t *out_accept_len, int32_t *out_commit_ids)
{
    t_err.clear();
    spec_status st = check_verify_args(target_logits, drafts, lanes, gamma, V, out_accept_len, out_commit_ids);
    if (st != SPEC_OK) return st;
    st = check_sampling(temperature, top_p, top_k, V, lanes, uniforms);
    if (st != SPEC_OK) return st;
    if (lanes == 0) return SPEC_OK;
    Sampling smp;
    smp.top_k = top_k;
    smp.temperature = temperature;
    smp.top_p = top_p;
    smp.uniforms = uniforms;
    return launch_round(nullptr, 0, 1, 1, nullptr, nullptr, nullptr, target_logits, drafts, lanes, gamma, V,
                        out_accept_len, out_commit_ids, nullptr, smp);
}

spec_status spec_verify(const uint16_t *target_logits, const int32_t *drafts, int64_t lanes, int32_t gamma,
                        int32_t *out_accept_len, int32_t *out_commit_ids)
{
    return spec_verify_v(target_logits, drafts, lanes, gamma, SPEC_VOCAB, out_accept_len, out_commit_ids);
}

spec_status spec_round(const uint16_t *draft_logits, int64_t cols, int64_t V, int32_t k, uint16_t *out_vals,
                       int32_t *out_ids, const uint16_t *target_logits, const int32_t *drafts, int64_t lanes,
                       int32_t gamma, int32_t *out_accept_len, int32_t *out_commit_ids)
{
    t_err.clear();
    spec_status st = check_topk_args(draft_logits, cols, V, k, out_vals, out_ids);
    if (st != SPEC_OK) return st;
    st = check_verify_args(target_logits, drafts, lanes, gamma, V, out_accept_len, out_commit_ids);
    if (st != SPEC_OK) return st;
    return launch_round(draft_logits, cols, V, k, nullptr, out_vals, out_ids, target_logits, drafts, lanes,
                        gamma, V, out_accept_len, out_commit_ids);
}

spec_status spec_round_counted(const uint16_t *draft_logits, int64_t cols, int64_t V, int32_t k,
                               uint16_t *out_vals, int32_t *out_ids, const uint16_t *target_logits,
                               const int32_t *drafts, int64_t lanes, int32_t gamma, int32_t *out_accept_len,
                               int32_t *out_commit_ids, spec_counters *counters)
{
    t_err.clear();
    spec_status st = check_topk_args(draft_logits, cols, V, k, out_vals, out_ids);
    if (st != SPEC_OK) return st;
    st = check_verify_args(target_logits, drafts, lanes, gamma, V, out_accept_len, out_commit_ids);
    if (st != SPEC_OK) return st;
    if (counters && misaligned(counters, 8)) return fail(SPEC_ERR_ARG, "counters misaligned (8 bytes needed)");
    return launch_round(draft_logits, cols, V, k, nullptr, out_vals, out_ids, target_logits, drafts, lanes,
                        gamma, V, out_accept_len, out_commit_ids, counters);
}

spec_status spec_round_host(const uint16_t *draft_logits, int64_t cols, int64_t V, int32_t k, uint16_t *out_vals,
                            int32_t *out_ids, const uint16_t *target_logits, const int32_t *drafts,
                            int64_t lanes, int32_t gamma, int32_t *out_accept_len, int32_t *out_commit_ids)
{
    t_err.clear();
    spec_status st = check_topk_args(draft_logits, cols, V, k, out_vals, out_ids);
    if (st != SPEC_OK) return st;
    st = check_verify_args(target_logits, drafts, lanes, gamma, V, out_accept_len, out_commit_ids);
    if (st != SPEC_OK) return st;
    if (cols == 0 && lanes == 0) return SPEC_OK;
    cudaStream_t stream = t_stream;
    if (stream_capturing(stream)) return fail(SPEC_ERR_ARG, "spec_round_host cannot be captured");
    const int64_t t_cols = lanes * (gamma + 1);
    const size_t b_dl = (size_t)cols * V * 2, b_tl = (size_t)t_cols * V * 2, b_dr = (size_t)lanes * gamma * 4;
    const size_t b_v = (size_t)cols * k * 2, b_i = (size_t)cols * k * 4, b_a = (size_t)lanes * 4,
                 b_c = (size_t)t_cols * 4;
    size_t off[7], tot = 0;
    const size_t sz[7] = {b_dl, b_tl, b_dr, b_v, b_i, b_a, b_c};
    for (int i = 0; i < 7; ++i) { off[i] = tot; tot = align256(tot + sz[i]); }
    // The lock is held from the staging lookup until the stream has drained:
    // host calls are serialised, so no other thread grows, frees or reuses
    // the staging area while this call's copies or kernel use it.
    std::lock_guard<std::mutex> lock(g_mu);
    DeviceState *d = nullptr;
    st = device_state(&d);
    if (st != SPEC_OK) return st;
    st = ensure_staging(*d, tot);
    if (st != SPEC_OK) return st;
    char *s = static_cast<char *>(d->staging);
    cudaError_t e = cudaSuccess;
    if (cols) e = cudaMemcpyAsync(s + off[0], draft_logits, b_dl, cudaMemcpyHostToDevice, stream);
    if (e == cudaSuccess && lanes) e = cudaMemcpyAsync(s + off[1], target_logits, b_tl, cudaMemcpyHostToDevice, stream);
    if (e == cudaSuccess && lanes) e = cudaMemcpyAsync(s + off[2], drafts, b_dr, cudaMemcpyHostToDevice, stream);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpyAsync H2D");
    st = launch_round_locked(cols ? (const uint16_t *)(s + off[0]) : nullptr, cols, V, k, nullptr,
                             cols ? (uint16_t *)(s + off[3]) : nullptr, cols ? (int32_t *)(s + off[4]) : nullptr,
                             lanes ? (const uint16_t *)(s + off[1]) : nullptr,
                             lanes ? (const int32_t *)(s + off[2]) : nullptr, lanes, gamma, V,
                             lanes ? (int32_t *)(s + off[5]) : nullptr, lanes ? (int32_t *)(s + off[6]) : nullptr);
    if (st != SPEC_OK) return st;
    if (cols) e = cudaMemcpyAsync(out_vals, s + off[3], b_v, cudaMemcpyDeviceToHost, stream);
    if (e == cudaSuccess && cols) e = cudaMemcpyAsync(out_ids, s + off[4], b_i, cudaMemcpyDeviceToHost, stream);
    if (e == cudaSuccess && lanes) e = cudaMemcpyAsync(out_accept_len, s + off[5], b_a, cudaMemcpyDeviceToHost, stream);
    if (e == cudaSuccess && lanes) e = cudaMemcpyAsync(out_commit_ids, s + off[6], b_c, cudaMemcpyDeviceToHost, stream);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpyAsync D2H");
    e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
    return SPEC_OK;
}

}  // extern "C"

// ---- the Q4 shortlist head ---------------------------------------------------

namespace {

spec_status check_head(int64_t rows, int64_t d, const void *wpack, const void *spack)
{
    if (rows < 16 || rows % 16 != 0 || rows > INT32_MAX)
        return fail(SPEC_ERR_ARG, "rows = %lld: need a positive multiple of 16 below 2^31", (long long)rows);
    if (d < 64 || d % 64 != 0 || d > q4::kMaxD)
        return fail(SPEC_ERR_ARG, "d = %lld: need a multiple of 64 in [64, %lld]", (long long)d, (long long)q4::kMaxD);
    if (!wpack || !spack) return fail(SPEC_ERR_ARG, "null pointer");
    if (misaligned(wpack, 16) || misaligned(spack, 4))
        return fail(SPEC_ERR_ARG, "misaligned packed head (weights need 16 bytes, scales 4)");
    return SPEC_OK;
}

// The head's logits for hidden states [cols][d] into logits [cols][rows],
// kColsPass hidden states per launch.  The caller holds g_mu.
spec_status launch_head_logits(const uint16_t *hidden, int64_t cols, int64_t d, const void *wpack, const void *spack,
                               int64_t rows, uint16_t *logits, cudaStream_t stream)
{
    DeviceState *dv = nullptr;
    spec_status st = device_state(&dv);
    if (st != SPEC_OK) return st;
    static bool attr_set[kMaxDevices] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (!attr_set[dev]) {
        cudaError_t e = cudaFuncSetAttribute(q4::logits_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)q4::smem_bytes(q4::kMaxD, 1));
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(q4::logits_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)q4::smem_bytes(q4::kMaxD, 2));
        if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute");
        attr_set[dev] = true;
    }
    const int64_t tiles = rows / 16;
    int64_t grid = (int64_t)dv->sms;
    const int64_t need = (tiles + q4::kWarps - 1) / q4::kWarps;
    if (grid > need) grid = need;
    for (int64_t c0 = 0; c0 < cols; c0 += q4::kColsPass) {
        cudaLaunchConfig_t cfg;
        memset(&cfg, 0, sizeof cfg);
        cfg.gridDim = dim3((unsigned)grid);
        cfg.blockDim = dim3(q4::kThreads);
        const int nt = cols - c0 > 8 ? 2 : 1;   // one n-tile when at most 8 hidden states are left
        cfg.dynamicSmemBytes = q4::smem_bytes(d, nt);
        cfg.stream = stream;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        const uint4 *w4 = static_cast<const uint4 *>(wpack);
        const uint32_t *s4 = static_cast<const uint32_t *>(spack);
        const cudaError_t e = nt == 2 ? cudaLaunchKernelEx(&cfg, q4::logits_kernel<2>, hidden, cols, d, w4, s4, rows, c0,
                                                           logits)
                                      : cudaLaunchKernelEx(&cfg, q4::logits_kernel<1>, hidden, cols, d, w4, s4, rows, c0,
                                                           logits);
        if (e != cudaSuccess) return cuda_fail(e, "kernel launch");
        g_launches.fetch_add(1, std::memory_order_relaxed);
    }
    return SPEC_OK;
}

}  // namespace

extern "C" {

spec_status spec_shortlist_pack(const uint8_t *weights, const uint16_t *scales, int64_t rows, int64_t d,
                                void *wpack, void *spack)
{
    t_err.clear();
    spec_status st = check_head(rows, d, wpack, spack);
    if (st != SPEC_OK) return st;
    if (!weights || !scales) return fail(SPEC_ERR_ARG, "null pointer");
    if (misaligned(scales, 2)) return fail(SPEC_ERR_ARG, "misaligned scales");
    std::lock_guard<std::mutex> lock(g_mu);
    DeviceState *dv = nullptr;
    st = device_state(&dv);
    if (st != SPEC_OK) return st;
    q4::pack_kernel<<<dv->sms * 4, 256, 0, t_stream>>>(weights, scales, rows, d, static_cast<uint32_t *>(wpack),
                                                         static_cast<uint32_t *>(spack));
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "kernel launch");
    g_launches.fetch_add(1, std::memory_order_relaxed);
    return SPEC_OK;
}

spec_status spec_shortlist_logits(const uint16_t *hidden, int64_t cols, int64_t d, const void *wpack,
                                  const void *spack, int64_t rows, uint16_t *out_logits)
{
    t_err.clear();
    if (cols < 0) return fail(SPEC_ERR_ARG, "cols = %lld < 0", (long long)cols);
    spec_status st = check_head(rows, d, wpack, spack);
    if (st != SPEC_OK) return st;
    if (cols == 0) return SPEC_OK;
    if (!hidden || !out_logits) return fail(SPEC_ERR_ARG, "null pointer");
    if (misaligned(hidden, 16) || misaligned(out_logits, 2))
        return fail(SPEC_ERR_ARG, "misaligned pointer (hidden states need 16 bytes, logits 2)");
    std::lock_guard<std::mutex> lock(g_mu);
    return launch_head_logits(hidden, cols, d, wpack, spack, rows, out_logits, t_stream);
}

spec_status spec_shortlist_topk(const uint16_t *hidden, int64_t cols, int64_t d, const void *wpack,
                                const void *spack, int64_t rows, const int32_t *id_map, int32_t k,
                                uint16_t *logits, uint16_t *out_vals, int32_t *out_ids)
{
    t_err.clear();
    if (cols < 0) return fail(SPEC_ERR_ARG, "cols = %lld < 0", (long long)cols);
    spec_status st = check_head(rows, d, wpack, spack);
    if (st != SPEC_OK) return st;
    st = check_topk_args(logits, cols, rows, k, out_vals, out_ids);
    if (st != SPEC_OK) return st;
    if (cols == 0) return SPEC_OK;
    if (!hidden || misaligned(hidden, 16)) return fail(SPEC_ERR_ARG, "hidden states null or misaligned (16 bytes)");
    if (!id_map || misaligned(id_map, 4)) return fail(SPEC_ERR_ARG, "id_map null or misaligned");
    std::lock_guard<std::mutex> lock(g_mu);
    st = launch_head_logits(hidden, cols, d, wpack, spack, rows, logits, t_stream);
    if (st != SPEC_OK) return st;
    return launch_round_locked(logits, cols, rows, k, id_map, out_vals, out_ids, nullptr, nullptr, 0, 1, 1, nullptr,
                               nullptr);
}

}  // extern "C"

extern "C" {

spec_status spec_set_kernel(int32_t which)
{
    t_err.clear();
    if (which != SPEC_KERNEL_AUTO && which != SPEC_KERNEL_WARP && which != SPEC_KERNEL_CTA &&
        which != SPEC_KERNEL_GROUPMAX)
        return fail(SPEC_ERR_ARG, "spec_set_kernel: unknown kernel %d", which);
    g_kernel_choice.store(which, std::memory_order_relaxed);
    return SPEC_OK;
}

int32_t spec_get_kernel(void) { return g_kernel_choice.load(std::memory_order_relaxed); }

int32_t spec_last_kernel(void) { return t_last_kernel; }

spec_status spec_set_stream(void *stream)
{
    t_stream = static_cast<cudaStream_t>(stream);
    return SPEC_OK;
}

void *spec_get_stream(void) { return static_cast<void *>(t_stream); }

spec_status spec_reserve(int64_t max_cols, int32_t max_k, int64_t max_lanes, int32_t max_gamma)
{
    t_err.clear();
    if (max_cols < 0 || max_lanes < 0 || max_k < 1 || max_k > SPEC_MAX_K || max_gamma < 1 ||
        max_gamma > SPEC_MAX_GAMMA)
        return fail(SPEC_ERR_ARG, "spec_reserve: bad sizes");
    std::lock_guard<std::mutex> lock(g_mu);
    DeviceState *d = nullptr;
    spec_status st = device_state(&d);
    if (st != SPEC_OK) return st;
    const int64_t t_cols = max_lanes * (max_gamma + 1);
    int occ = d->occ_w[0][0];
    for (int s = 0; s < 2; ++s)
        for (int m = 0; m < 2; ++m) occ = d->occ_w[s][m] > occ ? d->occ_w[s][m] : occ;
    const int64_t units = (int64_t)d->sms * occ * wrp::kWarpsPerCta;   // the per-warp kernel has the most units
    const ScratchCaps need = {2 * (max_cols + t_cols), max_lanes, units * 2 * (max_k + 2)};
    return ensure_scratch(*d, need, t_stream);
}

spec_status spec_release(void)
{
    t_err.clear();
    std::lock_guard<std::mutex> lock(g_mu);
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices) return SPEC_OK;
    DeviceState &d = g_dev[dev];
    if (!d.scratch && !d.staging && d.retired.empty()) return SPEC_OK;
    e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceSynchronize");
    if (d.scratch) cudaFree(d.scratch);
    if (d.staging) cudaFree(d.staging);
    for (void *p : d.retired) cudaFree(p);
    d.retired.clear();
    d.scratch = d.staging = nullptr;
    d.scratch_bytes = d.staging_bytes = 0;
    d.cap_cols = d.cap_lanes = d.cap_part = 0;
    return SPEC_OK;
}

const char *spec_last_error(void) { return t_err.c_str(); }

int64_t spec_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

spec_status spec_selftest_wait_timeout(int64_t limit_ns, uint64_t *out4)
{
    t_err.clear();
    if (limit_ns < 1000 || limit_ns > 1000000000) return fail(SPEC_ERR_ARG, "limit_ns outside [1 us, 1 s]");
    if (!out4 || misaligned(out4, 8)) return fail(SPEC_ERR_ARG, "out4 null or misaligned");
    wait_timeout_probe<<<1, 32, 0, t_stream>>>((uint64_t)limit_ns, reinterpret_cast<unsigned long long *>(out4));
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "kernel launch");
    return SPEC_OK;
}

spec_status spec_device_status(void)
{
    t_err.clear();
    cudaError_t e = cudaStreamSynchronize(t_stream);
    if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
    unsigned int flags = 0, zero = 0;
    e = cudaMemcpyFromSymbol(&flags, g_wait_timeouts, sizeof flags);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpyFromSymbol");
    if (flags == 0) return SPEC_OK;
    e = cudaMemcpyToSymbol(g_wait_timeouts, &zero, sizeof zero);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpyToSymbol");
    return fail(SPEC_ERR_CUDA, "a kernel gave up a bounded wait on its copy pipeline; its results are invalid");
}

}  // extern "C"

// ---------------------------------------------------------------------------
// spec_round_noalloc: the same round, with its scratch in a fixed device array
// ---------------------------------------------------------------------------
//
// Some callers cannot let this library call cudaMalloc: an inference engine
// that hands out every byte of device memory from its own pool (a stray
// allocation breaks its accounting and can fail once the pool has taken the
// free memory), a serving loop that must never pay the device-wide
// synchronisation that cudaFree implies, or a C host that runs under a fixed
// memory budget.  For them this entry point keeps its scratch (column and lane
// tickets, column certificates, partial lists) in one statically sized device
// array, so it allocates nothing, ever.  The array costs every GPU that loads
// the library its size until the process exits.

namespace {

constexpr int64_t kNoAllocMaxCols = SPEC_NOALLOC_MAX_COLS;     // draft + target columns
constexpr int64_t kNoAllocMaxLanes = SPEC_NOALLOC_MAX_LANES;
constexpr int64_t kNoAllocPartials = 131072;                    // partial-list entries (1 MiB)
constexpr size_t kNoAllocColTicket = 0;
constexpr size_t kNoAllocLaneTicket = kNoAllocColTicket + ((2 * kNoAllocMaxCols * 4 + 255) & ~int64_t(255));
constexpr size_t kNoAllocPart = kNoAllocLaneTicket + ((kNoAllocMaxLanes * 4 + 255) & ~int64_t(255));
constexpr size_t kNoAllocBytes = kNoAllocPart + kNoAllocPartials * 8;
constexpr size_t kNoAllocTicketBytes = kNoAllocPart;           // tickets and column certificates, cleared per call

// Device scratch of spec_round_noalloc.  In host code this name only stands
// for the symbol; the device address comes from cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocBytes];

void *g_noalloc_ptr[kMaxDevices] = {};

// Once per device, with that device current: look up the array's address.
spec_status noalloc_scratch(void **out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices) return fail(SPEC_ERR_CUDA, "device ordinal %d unsupported", dev);
    if (!g_noalloc_ptr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(static scratch)");
        g_noalloc_ptr[dev] = p;
    }
    *out = g_noalloc_ptr[dev];
    return SPEC_OK;
}

}  // namespace

extern "C" spec_status spec_round_noalloc(const uint16_t *draft_logits, int64_t cols, int64_t V, int32_t k,
                                          uint16_t *out_vals, int32_t *out_ids, const uint16_t *target_logits,
                                          const int32_t *drafts, int64_t lanes, int32_t gamma,
                                          int32_t *out_accept_len, int32_t *out_commit_ids)
{
    t_err.clear();
    spec_status st = check_topk_args(draft_logits, cols, V, k, out_vals, out_ids);
    if (st != SPEC_OK) return st;
    st = check_verify_args(target_logits, drafts, lanes, gamma, V, out_accept_len, out_commit_ids);
    if (st != SPEC_OK) return st;
    if (cols == 0 && lanes == 0) return SPEC_OK;
    // each term alone first: their sum could overflow for huge sizes
    if (cols > kNoAllocMaxCols || lanes > kNoAllocMaxLanes || lanes * (gamma + 1) > kNoAllocMaxCols - cols)
        return fail(SPEC_ERR_ARG, "spec_round_noalloc: %lld draft columns and %lld lanes of %d target columns "
                    "exceed its fixed scratch limits (%lld columns in all, %lld lanes)", (long long)cols,
                    (long long)lanes, gamma + 1, (long long)kNoAllocMaxCols, (long long)kNoAllocMaxLanes);
    const int64_t t_cols = lanes * (gamma + 1);

    std::lock_guard<std::mutex> lock(g_mu);
    DeviceState *d = nullptr;
    st = device_state(&d);
    if (st != SPEC_OK) return st;
    void *base = nullptr;
    st = noalloc_scratch(&base);
    if (st != SPEC_OK) return st;

    RoundArgs a;
    memset(&a, 0, sizeof a);
    a.draft = draft_logits; a.d_cols = cols; a.d_V = cols ? V : 1; a.k = cols ? k : 1;
    a.out_vals = out_vals; a.out_ids = out_ids;
    a.target = target_logits; a.t_cols = t_cols; a.t_V = lanes ? V : 1; a.gamma = gamma;
    a.drafts = drafts; a.out_accept = out_accept_len; a.out_commit = out_commit_ids;
    a.t_k = 1;   // greedy verify
    // units as in spec_round, fewer if their published lists would not fit
    const Plan plan = plan_round(*d, a, cols ? vectors_of(draft_logits, cols * V) : 0,
                                 lanes ? vectors_of(target_logits, t_cols * V) : 0, false, kNoAllocPartials);
    char *p = static_cast<char *>(base);
    a.col_ticket = reinterpret_cast<unsigned int *>(p + kNoAllocColTicket);
    a.col_cert = a.col_ticket + (cols + t_cols);
    a.lane_ticket = reinterpret_cast<unsigned int *>(p + kNoAllocLaneTicket);
    a.partials = reinterpret_cast<unsigned long long *>(p + kNoAllocPart);
    a.gkeys = reinterpret_cast<uint16_t *>(a.partials);

    cudaStream_t stream = t_stream;
    // the array keeps whatever the last call left: start every ticket at zero
    cudaError_t e = cudaMemsetAsync(base, 0, kNoAllocTicketBytes, stream);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync(static scratch tickets)");
    e = launch_plan(plan, a, stream, false);   // right after the ticket clear
    if (e != cudaSuccess) return cuda_fail(e, "kernel launch");
    g_launches.fetch_add(1, std::memory_order_relaxed);
    t_last_kernel = plan_kernel(plan);
    return SPEC_OK;
}
