// libspecsel: exact per-column top-k and fused greedy verify over bf16 logits
// for one GB300 (sm_103a).
//
// The operations ("A drafter inside the artifact", Ignis DFlash2 page,
// section "How it works"):
//   * top-k over each draft column of V logits: largest first, ties to the
//     smaller token id (third paragraph);
//   * greedy verify: per target column the argmax (same tie rule), then per
//     lane the longest run of drafts equal to those argmaxes, committed
//     together with the target's own next token (first paragraph).
//
// Design (one streaming pass over the logits, no tensor cores -- the step is
// a pure reduction bound by HBM bandwidth):
//   * Work units.  Every column is cut into P equal parts; a unit is one part
//     of one column.  A persistent grid of (SMs x resident CTAs) walks the
//     units round-robin.  P is chosen on the host so that the units spread
//     evenly over the CTAs (the pages' prior kernel gave one warp to each of
//     7 columns and sat 1,500x off its bandwidth floor).
//   * Inside a unit, the 8 warps take interleaved blocks of 256 16-byte
//     vectors (2,048 bf16); every lane issues its 8 vector loads before
//     looking at any of them.  A warp therefore walks its share of the unit
//     in increasing id order, which is what lets a tie with the running k-th
//     value be rejected without comparing ids.
//   * Per warp, the current top-k lives in registers, one (value, id) entry
//     per lane (two for k > 32).  A block is skipped after one bf16x2 max
//     tree and one compare against the running k-th value; only blocks with
//     a candidate take the slow path, which inserts candidates in id order
//     with a ballot/shuffle insertion.  The first block of a unit seeds the
//     threshold exactly from group maxima (the k-th largest of them, found
//     by a 16-step bisection on order-preserving keys), so the list fills
//     with ~k candidates instead of every element of the block.
//   * The 8 warp lists are merged in shared memory by rank (each entry
//     counts, by binary search, the better entries of the other lists).
//     If the column has several units, the CTA writes its list to scratch,
//     takes a ticket, and the last CTA to finish the column merges the
//     partial lists the same way -- no second pass over the logits, and no
//     spin-wait anywhere (nothing can hang).
//   * Verify columns are the k = 1 instance of the same path; the CTA that
//     finishes the last of a lane's gamma+1 columns runs the prefix match.
//   * Masked elements (outside the unit, or the ragged 16-byte edges of a
//     column) are bf16 NaN: bf16 max ignores them, ordered compares reject
//     them.  Edge vectors are read element by element, so no load ever
//     touches memory outside the caller's buffer.

#include <cuda_runtime.h>
#include <stdarg.h>
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include <atomic>
#include <mutex>
#include <string>

#include "specsel.h"

namespace {

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kU = 8;                       // 16-byte vectors per lane per block
constexpr int kBlockVec = 32 * kU;          // vectors per warp block (4 KiB)
constexpr int kListStride = 64;             // entries per list slot in shared memory
constexpr int kMaxParts = 32;               // parts per column (shared merge buffer)
constexpr int kMergeCap = 2048;             // entries in the shared merge buffer
constexpr unsigned kFull = 0xffffffffu;
constexpr uint32_t kNaN2 = 0x7FFF7FFFu;     // two bf16 NaNs: the mask value

static_assert(kWarps * kListStride <= kMergeCap, "warp lists must fit the merge buffer");
static_assert(kMaxParts * SPEC_MAX_K <= kMergeCap, "partials must fit the merge buffer");

struct RoundArgs {
    // top-k part (draft columns)
    const uint16_t *draft;
    int64_t d_cols, d_V;
    int32_t k, d_parts;
    const int32_t *id_map;
    uint16_t *out_vals;
    int32_t *out_ids;
    // verify part (target columns)
    const uint16_t *target;
    int64_t t_cols, t_V;
    int32_t t_parts, gamma;
    const int32_t *drafts;
    int32_t *out_accept;
    int32_t *out_commit;
    // scratch
    unsigned long long *partials;   // [n_units][pstride]
    unsigned int *col_ticket;       // [d_cols + t_cols]
    unsigned int *lane_ticket;      // [lanes]
    int32_t *t_argmax;              // [t_cols]
    int32_t pstride;
    int64_t d_units, n_units;
};

// ---------------------------------------------------------------------------
// device helpers
// ---------------------------------------------------------------------------

__device__ __forceinline__ uint4 ld_stream(const uint4 *p)
{
    uint4 r;
    asm("ld.global.nc.L1::no_allocate.L2::256B.v4.u32 {%0, %1, %2, %3}, [%4];"
        : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
        : "l"(p));
    return r;
}

__device__ __forceinline__ uint32_t bmax2(uint32_t a, uint32_t b)
{
    uint32_t d;
    asm("max.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// true if either bf16 half of a is > (or >=) the bf16 in both halves of t2;
// NaN halves compare false.
__device__ __forceinline__ bool any_gt(uint32_t a, uint32_t t2)
{
    uint32_t r;
    asm("{\n\t.reg .pred p, q;\n\t"
        "setp.gt.bf16x2 p|q, %1, %2;\n\t"
        "or.pred p, p, q;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(r)
        : "r"(a), "r"(t2));
    return r != 0;
}

__device__ __forceinline__ bool any_ge(uint32_t a, uint32_t t2)
{
    uint32_t r;
    asm("{\n\t.reg .pred p, q;\n\t"
        "setp.ge.bf16x2 p|q, %1, %2;\n\t"
        "or.pred p, p, q;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(r)
        : "r"(a), "r"(t2));
    return r != 0;
}

__device__ __forceinline__ float bf16_as_float(uint32_t raw16) { return __uint_as_float(raw16 << 16); }

// element e (0..7) of a 16-byte vector, widened exactly to float
__device__ __forceinline__ float elem8(const uint4 &q, int e)
{
    const uint32_t w = (e & 4) ? ((e & 2) ? q.w : q.z) : ((e & 2) ? q.y : q.x);
    return __uint_as_float((e & 1) ? (w & 0xFFFF0000u) : (w << 16));
}

// order-preserving 16-bit key of a bf16: -0 and +0 share a key; -Inf -> 0x80;
// NaN (the mask value) -> 0, below every real key.
__device__ __forceinline__ uint32_t order_key(uint32_t raw16)
{
    const uint32_t m = raw16 & 0x7FFFu;
    if (m > 0x7F80u) return 0u;
    return (raw16 & 0x8000u) ? (0x8000u - m) : (0x8000u + m);
}

__device__ __forceinline__ uint32_t key_to_raw(uint32_t key)
{
    const int s = (int)key - 0x8000;
    return s >= 0 ? (uint32_t)s : (0x8000u | (uint32_t)(-s));
}

// larger packed value = better entry: (key desc, id asc); low 16 bits keep the
// element's own bit pattern (so -0 survives); 0 = empty slot.
__device__ __forceinline__ unsigned long long pack_entry(float v, uint32_t id)
{
    if (v != v) return 0ull;
    const uint32_t raw = __float_as_uint(v) >> 16;
    return ((unsigned long long)order_key(raw) << 48) | ((unsigned long long)(~id) << 16) | raw;
}

__device__ __forceinline__ uint32_t entry_id(unsigned long long e) { return ~(uint32_t)(e >> 16); }
__device__ __forceinline__ uint16_t entry_raw(unsigned long long e) { return (uint16_t)(e & 0xFFFFu); }

// bf16x2 max over one 16-byte vector
__device__ __forceinline__ uint32_t vmax(const uint4 &q) { return bmax2(bmax2(q.x, q.y), bmax2(q.z, q.w)); }

// both halves hold max(lo, hi)
__device__ __forceinline__ uint32_t hmax_splat(uint32_t m2) { return bmax2(m2, __byte_perm(m2, 0, 0x1032)); }

// Masked load of an edge vector: element by element, only inside [g0, g1).
__device__ __forceinline__ uint4 load_edge(const uint16_t *buf, int64_t j, int mis, int64_t g0, int64_t g1)
{
    uint32_t w[4];
#pragma unroll
    for (int h = 0; h < 4; ++h) {
        uint32_t lo = 0x7FFFu, hi = 0x7FFFu;
        const int64_t ga = 8 * j + 2 * h - mis, gb = ga + 1;
        if (ga >= g0 && ga < g1) lo = __ldg(buf + ga);
        if (gb >= g0 && gb < g1) hi = __ldg(buf + gb);
        w[h] = lo | (hi << 16);
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
}

// Insert candidate (cv, cid) into the warp-distributed sorted list.  Entry
// index s*32+lane lives in Lv[s]/Li[s].  Without an id map, candidates reach
// the list in increasing id order, so an equal value already in the list is
// better; with an id map, ties compare the mapped ids.
template <int SLOTS, bool MAPPED>
__device__ __forceinline__ void list_insert(float (&Lv)[SLOTS], uint32_t (&Li)[SLOTS], float cv,
                                            uint32_t cid, int kk, int lane)
{
    int pos = 0;
#pragma unroll
    for (int s = 0; s < SLOTS; ++s) {
        bool better = MAPPED ? (Lv[s] > cv || (Lv[s] == cv && Li[s] < cid)) : (Lv[s] >= cv);
        better = better && (s * 32 + lane < kk);
        pos += __popc(__ballot_sync(kFull, better));
    }
    if (pos >= kk) return;
    const float up0 = __shfl_up_sync(kFull, Lv[0], 1);
    const uint32_t ui0 = __shfl_up_sync(kFull, Li[0], 1);
    if constexpr (SLOTS == 2) {
        const float last0 = __shfl_sync(kFull, Lv[0], 31);
        const uint32_t lasti0 = __shfl_sync(kFull, Li[0], 31);
        float up1 = __shfl_up_sync(kFull, Lv[1], 1);
        uint32_t ui1 = __shfl_up_sync(kFull, Li[1], 1);
        if (lane == 0) { up1 = last0; ui1 = lasti0; }
        const int i1 = 32 + lane;
        if (i1 > pos) { Lv[1] = up1; Li[1] = ui1; }
        else if (i1 == pos) { Lv[1] = cv; Li[1] = cid; }
    }
    if (lane > pos) { Lv[0] = up0; Li[0] = ui0; }
    else if (lane == pos) { Lv[0] = cv; Li[0] = cid; }
}

template <int SLOTS>
__device__ __forceinline__ float list_kth(const float (&Lv)[SLOTS], int kk)
{
    const int i = kk - 1;
    float t = __shfl_sync(kFull, Lv[0], i & 31);
    if constexpr (SLOTS == 2) {
        const float t1 = __shfl_sync(kFull, Lv[1], i & 31);
        if (i >= 32) t = t1;
    }
    return t;
}

// Loads one warp block (kU vectors per lane) of the unit: interior vectors
// with 16-byte loads, the unit's two edge vectors element by element, and
// vectors past the unit as masked NaNs.
__device__ __forceinline__ void load_block(uint4 (&x)[kU], const uint16_t *__restrict__ buf, const uint4 *vb,
                                           int64_t jb, int64_t jf, int64_t jl, int mis, int64_t g0, int64_t g1,
                                           int lane)
{
    if (jb > jf && jb + kBlockVec - 1 < jl) {
#pragma unroll
        for (int u = 0; u < kU; ++u) x[u] = ld_stream(vb + jb + u * 32 + lane);
    } else {
#pragma unroll
        for (int u = 0; u < kU; ++u) {
            const int64_t j = jb + u * 32 + lane;
            if (j > jf && j < jl) x[u] = ld_stream(vb + j);
            else if (j == jf || j == jl) x[u] = load_edge(buf, j, mis, g0, g1);
            else x[u] = make_uint4(kNaN2, kNaN2, kNaN2, kNaN2);
        }
    }
}

// Threshold of a list: kk entries >= it exist (a certificate).  Candidates
// must be >= `thr` (inclusive) or, when `strict`, > `thr`.
struct Threshold {
    float thr;
    uint32_t thr2;   // thr as a bf16 pair
    bool strict;
};

__device__ __forceinline__ Threshold make_threshold(uint32_t cta_key, float own, bool own_full, bool mapped)
{
    // cta_key: order key certified for the whole CTA (0 = none yet)
    Threshold t;
    const uint32_t own_key = own_full ? order_key(__float_as_uint(own) >> 16) : 0u;
    if (own_full && own_key >= cta_key) {
        t.thr = own;
        t.strict = !mapped;
    } else {
        t.thr = cta_key ? bf16_as_float(key_to_raw(cta_key)) : -INFINITY;
        t.strict = false;
    }
    const uint32_t raw = __float_as_uint(t.thr) >> 16;
    t.thr2 = raw | (raw << 16);
    return t;
}

// One warp's pass over its blocks of one unit; leaves its list (packed,
// sorted, empty slots = 0) in lists[warp * kListStride + i], i < kk.
//
// The CTA shares one threshold key in *cta_thr: whenever a warp's list is
// full, its kk-th value certifies kk elements of the unit at or above it, so
// no element below it can be in the unit's top-k.  Every warp filters
// against the larger of that key and its own list's kk-th value (strictly,
// for its own value: the warp sees its elements in id order, so an equal
// value arriving later has the larger id).  All threads of the CTA must
// call this (it contains one CTA barrier); *cta_thr must be 0 on entry.
template <int SLOTS, bool MAPPED>
__device__ __forceinline__ void scan_unit(const uint16_t *__restrict__ buf, int64_t V, int64_t col,
                                          int64_t e0, int64_t e1, int kk,
                                          const int32_t *__restrict__ id_map,
                                          unsigned long long *lists, unsigned int *cta_thr)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(buf);
    const int mis = (int)((a0 >> 1) & 7);                      // element phase of buf in 16 B
    const uint4 *vb = reinterpret_cast<const uint4 *>(a0 - 2 * (uintptr_t)mis);
    const int64_t colbase = col * V;
    const int64_t g0 = colbase + e0, g1 = colbase + e1;       // element range in buf
    const int64_t jf = (g0 + mis) >> 3, jl = (g1 - 1 + mis) >> 3;
    const int64_t nblk = (jl - jf + kBlockVec) / kBlockVec;

    float Lv[SLOTS];
    uint32_t Li[SLOTS];
#pragma unroll
    for (int s = 0; s < SLOTS; ++s) { Lv[s] = __uint_as_float(0x7FC00000u); Li[s] = 0xFFFFFFFFu; }
    bool full = false;
    volatile unsigned int *vthr = cta_thr;

    // Seed: from its first block each warp certifies the kk-th largest of
    // its group maxima (kk distinct elements are at or above it); the CTA
    // keeps the largest certificate.
    uint4 x[kU];
    int64_t b = warp;
    if (b < nblk) {
        load_block(x, buf, vb, jf + b * kBlockVec, jf, jl, mis, g0, g1, lane);
        constexpr int G = (SLOTS == 1) ? 1 : 4;
        constexpr int PER = kU / G;
        uint32_t key[G];
#pragma unroll
        for (int g = 0; g < G; ++g) {
            uint32_t m = vmax(x[g * PER]);
#pragma unroll
            for (int u = 1; u < PER; ++u) m = bmax2(m, vmax(x[g * PER + u]));
            key[g] = order_key(hmax_splat(m) & 0xFFFFu);
        }
        uint32_t t = 0;
        if (kk == 1) {
            t = __reduce_max_sync(kFull, key[0]);
        } else {
#pragma unroll 1
            for (int bit = 15; bit >= 0; --bit) {
                const uint32_t tr = t | (1u << bit);
                int cnt = 0;
#pragma unroll
                for (int g = 0; g < G; ++g) cnt += __popc(__ballot_sync(kFull, key[g] >= tr));
                if (cnt >= kk) t = tr;
            }
        }
        if (lane == 0 && t != 0) atomicMax(cta_thr, t);
    }
    __syncthreads();

    for (; b < nblk; b += kWarps) {
        const int64_t jb = jf + b * kBlockVec;
        if (b != warp) load_block(x, buf, vb, jb, jf, jl, mis, g0, g1, lane);
        const Threshold T = make_threshold(*vthr, list_kth<SLOTS>(Lv, kk), full, MAPPED);

        uint32_t m = vmax(x[0]);
#pragma unroll
        for (int u = 1; u < kU; ++u) m = bmax2(m, vmax(x[u]));
        const bool pass = T.strict ? any_gt(m, T.thr2) : any_ge(m, T.thr2);
        if (!__ballot_sync(kFull, pass)) continue;

        // Slow path: insert this block's candidates in increasing id order
        // (vector u, then lane, then element).
        const int64_t id_lane = 8 * (jb + lane) - mis - colbase;   // id of element 0, vector 0
#pragma unroll
        for (int u = 0; u < kU; ++u) {
            const bool pu = pass && (T.strict ? any_gt(vmax(x[u]), T.thr2) : any_ge(vmax(x[u]), T.thr2));
            if (!__ballot_sync(kFull, pu)) continue;
            uint32_t cm = 0;
            if (pu) {
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const float v = elem8(x[u], e);
                    cm |= (uint32_t)(T.strict ? (v > T.thr) : (v >= T.thr)) << e;
                }
            }
            uint32_t act = __ballot_sync(kFull, cm != 0);
            while (act) {
                const int src = __ffs(act) - 1;
                float cv = 0.f;
                uint32_t cid = 0;
                if (lane == src) {
                    const int e = __ffs(cm) - 1;
                    cm &= cm - 1;
                    cv = elem8(x[u], e);
                    cid = (uint32_t)(id_lane + 256 * u + e);
                    if (MAPPED) cid = (uint32_t)__ldg(id_map + cid);
                }
                cv = __shfl_sync(kFull, cv, src);
                cid = __shfl_sync(kFull, cid, src);
                list_insert<SLOTS, MAPPED>(Lv, Li, cv, cid, kk, lane);
                act = __ballot_sync(kFull, cm != 0);
            }
        }
        const float tv = list_kth<SLOTS>(Lv, kk);
        full = (tv == tv);
        if (full && lane == 0) {
            const uint32_t kkey = order_key(__float_as_uint(tv) >> 16);
            if (kkey > *vthr) atomicMax(cta_thr, kkey);
        }
    }

#pragma unroll
    for (int s = 0; s < SLOTS; ++s) {
        const int i = s * 32 + lane;
        if (i < kk) lists[warp * kListStride + i] = pack_entry(Lv[s], Li[s]);
    }
}

// out[0..kk) = the kk best of nl sorted lists (stride apart, kk long, empty
// slots 0 at the tail).  Caller zeroes out and synchronises around the call.
__device__ __forceinline__ void rank_merge(const unsigned long long *lists, int nl, int stride, int kk,
                                           unsigned long long *out)
{
    for (int idx = threadIdx.x; idx < nl * kk; idx += blockDim.x) {
        const int li = idx / kk, r = idx - li * kk;
        const unsigned long long e = lists[li * stride + r];
        if (e == 0ull) continue;
        int rank = r;
        for (int o = 0; o < nl && rank < kk; ++o) {
            if (o == li) continue;
            const unsigned long long *L = lists + o * stride;
            int lo = 0, hi = kk;
            while (lo < hi) {
                const int mid = (lo + hi) >> 1;
                if (L[mid] > e) lo = mid + 1;
                else hi = mid;
            }
            rank += lo;
        }
        if (rank < kk) out[rank] = e;
    }
}

struct Shared {
    unsigned long long buf[kMergeCap];
    unsigned long long out[SPEC_MAX_K];
    unsigned int thr;   // CTA-wide certified threshold key of the current unit
    int flag;
};

// A column's final list is in s.out[0..kk): write the top-k outputs, or, for
// a target column, record its argmax and run the lane's prefix match if this
// was the lane's last column.
__device__ __forceinline__ void finish_column(const RoundArgs &a, bool draft, int64_t col, int kk,
                                              const Shared &s)
{
    if (draft) {
        for (int i = threadIdx.x; i < kk; i += blockDim.x) {
            const unsigned long long e = s.out[i];
            a.out_vals[col * kk + i] = entry_raw(e);
            a.out_ids[col * kk + i] = (int32_t)entry_id(e);
        }
        return;
    }
    if (threadIdx.x != 0) return;
    const int gp1 = a.gamma + 1;
    const int64_t lane = col / gp1;
    a.t_argmax[col] = (int32_t)entry_id(s.out[0]);
    __threadfence();
    const unsigned old = atomicAdd(a.lane_ticket + lane, 1u);
    if (old != (unsigned)a.gamma) return;
    __threadfence();
    const int32_t *ta = a.t_argmax + lane * gp1;
    const int32_t *dr = a.drafts + lane * a.gamma;
    int acc = 0;
    while (acc < a.gamma && __ldg(dr + acc) == __ldcg(ta + acc)) ++acc;
    a.out_accept[lane] = acc;
    for (int j = 0; j < gp1; ++j) a.out_commit[lane * gp1 + j] = (j <= acc) ? __ldcg(ta + j) : -1;
    a.lane_ticket[lane] = 0u;   // ready for the next launch
}

template <int SLOTS, bool MAPPED>
__global__ void __launch_bounds__(kThreads, 2) spec_round_kernel(const RoundArgs a)
{
    __shared__ Shared s;
    for (int64_t u = blockIdx.x; u < a.n_units; u += gridDim.x) {
        const bool draft = u < a.d_units;
        const int64_t v = draft ? u : u - a.d_units;
        const int parts = draft ? a.d_parts : a.t_parts;
        const int64_t V = draft ? a.d_V : a.t_V;
        const int64_t col = v / parts;
        const int p = (int)(v - col * parts);
        const int64_t e0 = (int64_t)p * V / parts, e1 = (int64_t)(p + 1) * V / parts;
        const int kk = draft ? a.k : 1;

        if (threadIdx.x == 0) s.thr = 0u;      // nobody reads it past the last unit's scan
        __syncthreads();                       // previous unit's use of s is over
        if (draft) scan_unit<SLOTS, MAPPED>(a.draft, V, col, e0, e1, kk, a.id_map, s.buf, &s.thr);
        else scan_unit<1, false>(a.target, V, col, e0, e1, 1, nullptr, s.buf, &s.thr);
        for (int i = threadIdx.x; i < kk; i += blockDim.x) s.out[i] = 0ull;
        __syncthreads();
        rank_merge(s.buf, kWarps, kListStride, kk, s.out);
        __syncthreads();

        if (parts == 1) {
            finish_column(a, draft, col, kk, s);
            continue;
        }
        // several units per column: publish, take a ticket, last one merges
        unsigned long long *mine = a.partials + u * a.pstride;
        for (int i = threadIdx.x; i < kk; i += blockDim.x) mine[i] = s.out[i];
        __threadfence();
        __syncthreads();
        const int64_t tix = draft ? col : a.d_cols + col;
        if (threadIdx.x == 0) s.flag = (atomicAdd(a.col_ticket + tix, 1u) == (unsigned)(parts - 1));
        __syncthreads();
        if (!s.flag) continue;
        __threadfence();
        const unsigned long long *first = a.partials + (u - p) * a.pstride;
        for (int idx = threadIdx.x; idx < parts * kk; idx += blockDim.x) {
            const int li = idx / kk, r = idx - li * kk;
            s.buf[idx] = __ldcg(first + (int64_t)li * a.pstride + r);
        }
        for (int i = threadIdx.x; i < kk; i += blockDim.x) s.out[i] = 0ull;
        __syncthreads();
        rank_merge(s.buf, parts, kk, kk, s.out);
        __syncthreads();
        finish_column(a, draft, col, kk, s);
        if (threadIdx.x == 0) a.col_ticket[tix] = 0u;   // ready for the next launch
    }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------

constexpr int kMaxDevices = 64;

struct DeviceState {
    bool init = false;
    int sms = 0;
    int occ[2][2] = {{0, 0}, {0, 0}};   // resident CTAs per SM, [slots-1][mapped]
    // Scratch: [col tickets | lane tickets | target argmax | partial lists].
    // Each region keeps its place and capacity until the whole area is
    // reallocated (and zeroed), so a ticket is never laid over stale data.
    void *scratch = nullptr;
    size_t scratch_bytes = 0;
    int64_t cap_cols = 0, cap_lanes = 0, cap_tcols = 0, cap_part = 0;
    void *staging = nullptr;
    size_t staging_bytes = 0;
};

std::mutex g_mu;
DeviceState g_dev[kMaxDevices];
std::atomic<int64_t> g_launches{0};
thread_local cudaStream_t t_stream = nullptr;
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
void *kernel_ptr() { return reinterpret_cast<void *>(spec_round_kernel<S, M>); }

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
        void *kp[2][2] = {{kernel_ptr<1, false>(), kernel_ptr<1, true>()},
                          {kernel_ptr<2, false>(), kernel_ptr<2, true>()}};
        for (int s = 0; s < 2; ++s)
            for (int m = 0; m < 2; ++m) {
                e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&d.occ[s][m], kp[s][m], kThreads, 0);
                if (e != cudaSuccess) return cuda_fail(e, "cudaOccupancyMaxActiveBlocksPerMultiprocessor");
                if (d.occ[s][m] < 1) d.occ[s][m] = 1;
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
    int32_t *t_argmax;
    unsigned long long *partials;
};

struct ScratchCaps {
    int64_t cols, lanes, tcols, part;   // part = partial-list entries (u64)
};

size_t scratch_bytes(const ScratchCaps &c)
{
    return align256((size_t)c.cols * 4) + align256((size_t)c.lanes * 4) + align256((size_t)c.tcols * 4) +
           align256((size_t)c.part * 8);
}

ScratchPtrs scratch_ptrs(const DeviceState &d)
{
    char *p = static_cast<char *>(d.scratch);
    ScratchPtrs s;
    s.col_ticket = reinterpret_cast<unsigned int *>(p);
    p += align256((size_t)d.cap_cols * 4);
    s.lane_ticket = reinterpret_cast<unsigned int *>(p);
    p += align256((size_t)d.cap_lanes * 4);
    s.t_argmax = reinterpret_cast<int32_t *>(p);
    p += align256((size_t)d.cap_tcols * 4);
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
// when they finish.
spec_status ensure_scratch(DeviceState &d, const ScratchCaps &need, cudaStream_t st)
{
    if (d.scratch && need.cols <= d.cap_cols && need.lanes <= d.cap_lanes && need.tcols <= d.cap_tcols &&
        need.part <= d.cap_part)
        return SPEC_OK;
    if (stream_capturing(st))
        return fail(SPEC_ERR_ALLOC, "scratch must grow during stream capture; call spec_reserve before capturing");
    auto grow = [](int64_t have, int64_t want) { return want <= have ? have : want + want / 4 + 64; };
    ScratchCaps c;
    c.cols = grow(d.cap_cols, need.cols);
    c.lanes = grow(d.cap_lanes, need.lanes);
    c.tcols = grow(d.cap_tcols, need.tcols);
    c.part = grow(d.cap_part, need.part);
    const size_t bytes = scratch_bytes(c);
    cudaError_t e;
    if (d.scratch) {
        e = cudaDeviceSynchronize();
        if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceSynchronize");
        cudaFree(d.scratch);
        d.scratch = nullptr;
        d.scratch_bytes = 0;
        d.cap_cols = d.cap_lanes = d.cap_tcols = d.cap_part = 0;
    }
    e = cudaMalloc(&d.scratch, bytes);
    if (e != cudaSuccess) {
        d.scratch = nullptr;
        cudaGetLastError();
        return fail(SPEC_ERR_ALLOC, "cudaMalloc(%zu) for scratch: %s", bytes, cudaGetErrorString(e));
    }
    e = cudaMemset(d.scratch, 0, bytes);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemset scratch");
    d.scratch_bytes = bytes;
    d.cap_cols = c.cols;
    d.cap_lanes = c.lanes;
    d.cap_tcols = c.tcols;
    d.cap_part = c.part;
    return SPEC_OK;
}

// Choose the number of parts per column: minimise the slowest CTA's work
// (units are handed out round-robin), counting a fixed cost per unit and
// per cross-CTA merge, in element-equivalents.
int choose_parts(int64_t n_cols, int64_t V, int64_t max_ctas)
{
    const int64_t kUnitCost = 3000, kMergeCost = 6000;
    int64_t pmax = V / 2048;
    if (pmax < 1) pmax = 1;
    if (pmax > kMaxParts) pmax = kMaxParts;
    int best = 1;
    int64_t best_cost = INT64_MAX;
    for (int64_t P = 1; P <= pmax; ++P) {
        const int64_t units = n_cols * P;
        const int64_t ctas = units < max_ctas ? units : max_ctas;
        const int64_t rounds = (units + ctas - 1) / ctas;
        const int64_t cost = rounds * ((V + P - 1) / P + kUnitCost) + (P > 1 ? kMergeCost : 0);
        if (cost < best_cost) { best_cost = cost; best = (int)P; }
    }
    return best;
}

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
spec_status launch_round(const uint16_t *draft, int64_t cols, int64_t V, int32_t k, const int32_t *id_map,
                         uint16_t *vals, int32_t *ids, const uint16_t *target, const int32_t *drafts,
                         int64_t lanes, int32_t gamma, int64_t tV, int32_t *acc, int32_t *com)
{
    if (cols == 0 && lanes == 0) return SPEC_OK;
    std::lock_guard<std::mutex> lock(g_mu);
    DeviceState *d = nullptr;
    spec_status st = device_state(&d);
    if (st != SPEC_OK) return st;
    const int slots = (cols > 0 && k > 32) ? 2 : 1;
    const bool mapped = cols > 0 && id_map != nullptr;
    const int64_t max_ctas = (int64_t)d->sms * d->occ[slots - 1][mapped ? 1 : 0];
    const int64_t t_cols = lanes * (gamma + 1);

    RoundArgs a;
    memset(&a, 0, sizeof a);
    a.draft = draft; a.d_cols = cols; a.d_V = cols ? V : 1; a.k = cols ? k : 1;
    a.id_map = id_map; a.out_vals = vals; a.out_ids = ids;
    a.target = target; a.t_cols = t_cols; a.t_V = lanes ? tV : 1; a.gamma = gamma;
    a.drafts = drafts; a.out_accept = acc; a.out_commit = com;
    if (cols > 0 && lanes > 0 && V == tV) {
        a.d_parts = a.t_parts = choose_parts(cols + t_cols, V, max_ctas);
    } else {
        a.d_parts = cols ? choose_parts(cols, V, max_ctas) : 1;
        a.t_parts = lanes ? choose_parts(t_cols, tV, max_ctas) : 1;
    }
    a.d_units = cols * a.d_parts;
    a.n_units = a.d_units + t_cols * a.t_parts;
    a.pstride = a.k;
    cudaStream_t stream = t_stream;
    const ScratchCaps need = {cols + t_cols, lanes, t_cols, a.n_units * a.pstride};
    st = ensure_scratch(*d, need, stream);
    if (st != SPEC_OK) return st;
    const ScratchPtrs sp = scratch_ptrs(*d);
    a.partials = sp.partials;
    a.col_ticket = sp.col_ticket;
    a.lane_ticket = sp.lane_ticket;
    a.t_argmax = sp.t_argmax;

    const int64_t grid64 = a.n_units < max_ctas ? a.n_units : max_ctas;
    const dim3 grid((unsigned)grid64), block(kThreads);
    if (slots == 1 && !mapped) spec_round_kernel<1, false><<<grid, block, 0, stream>>>(a);
    else if (slots == 1) spec_round_kernel<1, true><<<grid, block, 0, stream>>>(a);
    else if (!mapped) spec_round_kernel<2, false><<<grid, block, 0, stream>>>(a);
    else spec_round_kernel<2, true><<<grid, block, 0, stream>>>(a);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "kernel launch");
    g_launches.fetch_add(1, std::memory_order_relaxed);
    return SPEC_OK;
}

spec_status ensure_staging(DeviceState &d, size_t bytes)
{
    if (d.staging_bytes >= bytes) return SPEC_OK;
    cudaError_t e;
    if (d.staging) {
        e = cudaDeviceSynchronize();
        if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceSynchronize");
        cudaFree(d.staging);
        d.staging = nullptr;
        d.staging_bytes = 0;
    }
    e = cudaMalloc(&d.staging, bytes);
    if (e != cudaSuccess) {
        d.staging = nullptr;
        cudaGetLastError();
        return fail(SPEC_ERR_ALLOC, "cudaMalloc(%zu) for staging: %s", bytes, cudaGetErrorString(e));
    }
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
    char *s = nullptr;
    {
        std::lock_guard<std::mutex> lock(g_mu);
        DeviceState *d = nullptr;
        st = device_state(&d);
        if (st != SPEC_OK) return st;
        st = ensure_staging(*d, tot);
        if (st != SPEC_OK) return st;
        s = static_cast<char *>(d->staging);
    }
    cudaError_t e = cudaSuccess;
    if (cols) e = cudaMemcpyAsync(s + off[0], draft_logits, b_dl, cudaMemcpyHostToDevice, stream);
    if (e == cudaSuccess && lanes) e = cudaMemcpyAsync(s + off[1], target_logits, b_tl, cudaMemcpyHostToDevice, stream);
    if (e == cudaSuccess && lanes) e = cudaMemcpyAsync(s + off[2], drafts, b_dr, cudaMemcpyHostToDevice, stream);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpyAsync H2D");
    st = spec_round(cols ? (const uint16_t *)(s + off[0]) : nullptr, cols, V, k,
                    cols ? (uint16_t *)(s + off[3]) : nullptr, cols ? (int32_t *)(s + off[4]) : nullptr,
                    lanes ? (const uint16_t *)(s + off[1]) : nullptr, lanes ? (const int32_t *)(s + off[2]) : nullptr,
                    lanes, gamma, lanes ? (int32_t *)(s + off[5]) : nullptr, lanes ? (int32_t *)(s + off[6]) : nullptr);
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
    const ScratchCaps need = {max_cols + t_cols, max_lanes, t_cols, (max_cols + t_cols) * kMaxParts * max_k};
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
    if (!d.scratch && !d.staging) return SPEC_OK;
    e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceSynchronize");
    if (d.scratch) cudaFree(d.scratch);
    if (d.staging) cudaFree(d.staging);
    d.scratch = d.staging = nullptr;
    d.scratch_bytes = d.staging_bytes = 0;
    d.cap_cols = d.cap_lanes = d.cap_tcols = d.cap_part = 0;
    return SPEC_OK;
}

const char *spec_last_error(void) { return t_err.c_str(); }

int64_t spec_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

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
// tickets, target argmaxes, partial lists) in one statically sized device
// array, so it allocates nothing, ever.  The array costs every GPU that loads
// the library its size until the process exits.

namespace {

constexpr int64_t kNoAllocMaxCols = SPEC_NOALLOC_MAX_COLS;     // draft + target columns
constexpr int64_t kNoAllocMaxLanes = SPEC_NOALLOC_MAX_LANES;
constexpr int64_t kNoAllocPartials = 131072;                    // partial-list entries (1 MiB)
constexpr size_t kNoAllocColTicket = 0;
constexpr size_t kNoAllocLaneTicket = kNoAllocColTicket + ((kNoAllocMaxCols * 4 + 255) & ~int64_t(255));
constexpr size_t kNoAllocArgmax = kNoAllocLaneTicket + ((kNoAllocMaxLanes * 4 + 255) & ~int64_t(255));
constexpr size_t kNoAllocPart = kNoAllocArgmax + ((kNoAllocMaxCols * 4 + 255) & ~int64_t(255));
constexpr size_t kNoAllocBytes = kNoAllocPart + kNoAllocPartials * 8;
constexpr size_t kNoAllocTicketBytes = kNoAllocArgmax;         // both ticket arrays, cleared per call

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
    const int64_t t_cols = lanes * (gamma + 1);
    if (cols + t_cols > kNoAllocMaxCols)
        return fail(SPEC_ERR_ARG, "spec_round_noalloc: %lld draft + target columns exceed its fixed scratch "
                    "limit of %lld", (long long)(cols + t_cols), (long long)kNoAllocMaxCols);
    if (lanes > kNoAllocMaxLanes)
        return fail(SPEC_ERR_ARG, "spec_round_noalloc: %lld lanes exceed its fixed scratch limit of %lld",
                    (long long)lanes, (long long)kNoAllocMaxLanes);

    std::lock_guard<std::mutex> lock(g_mu);
    DeviceState *d = nullptr;
    st = device_state(&d);
    if (st != SPEC_OK) return st;
    void *base = nullptr;
    st = noalloc_scratch(&base);
    if (st != SPEC_OK) return st;

    const int slots = (cols > 0 && k > 32) ? 2 : 1;
    const int64_t max_ctas = (int64_t)d->sms * d->occ[slots - 1][0];
    RoundArgs a;
    memset(&a, 0, sizeof a);
    a.draft = draft_logits; a.d_cols = cols; a.d_V = cols ? V : 1; a.k = cols ? k : 1;
    a.out_vals = out_vals; a.out_ids = out_ids;
    a.target = target_logits; a.t_cols = t_cols; a.t_V = lanes ? V : 1; a.gamma = gamma;
    a.drafts = drafts; a.out_accept = out_accept_len; a.out_commit = out_commit_ids;
    a.pstride = a.k;
    // parts per column as in spec_round, capped so the partial lists fit
    int parts = choose_parts(cols + t_cols, V, max_ctas);
    const int64_t cap = kNoAllocPartials / ((cols + t_cols) * (int64_t)a.pstride);
    if (parts > cap) parts = cap < 1 ? 1 : (int)cap;        // one part per column needs no partials
    a.d_parts = a.t_parts = parts;
    a.d_units = cols * parts;
    a.n_units = a.d_units + t_cols * parts;
    char *p = static_cast<char *>(base);
    a.col_ticket = reinterpret_cast<unsigned int *>(p + kNoAllocColTicket);
    a.lane_ticket = reinterpret_cast<unsigned int *>(p + kNoAllocLaneTicket);
    a.t_argmax = reinterpret_cast<int32_t *>(p + kNoAllocArgmax);
    a.partials = reinterpret_cast<unsigned long long *>(p + kNoAllocPart);

    cudaStream_t stream = t_stream;
    // the array keeps whatever the last call left: start every ticket at zero
    cudaError_t e = cudaMemsetAsync(base, 0, kNoAllocTicketBytes, stream);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync(static scratch tickets)");
    const int64_t grid64 = a.n_units < max_ctas ? a.n_units : max_ctas;
    const dim3 grid((unsigned)grid64), block(kThreads);
    if (slots == 1) spec_round_kernel<1, false><<<grid, block, 0, stream>>>(a);
    else spec_round_kernel<2, false><<<grid, block, 0, stream>>>(a);
    e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "kernel launch");
    g_launches.fetch_add(1, std::memory_order_relaxed);
    return SPEC_OK;
}
