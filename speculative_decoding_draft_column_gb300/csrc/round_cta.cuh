// The CTA-cooperative streaming kernel (small rounds): one CTA per SM owns
// a contiguous slice of the flat run of logits and streams it in 60 KiB
// chunks through a three-chunk shared-memory ring (bulk copies completing on
// mbarriers).  Fifteen warps filter a 4 KiB share of every chunk each against
// the column's certificate and append their candidates; a sixteenth warp
// folds them into the CTA's sorted list for the column, publishes the list's
// kk-th key as the new certificate, and finishes columns (emit, or publish
// and merge across CTAs; verify's prefix match on a lane's last column).
// Every column thus has one threshold per CTA -- the kk-th best of all that
// CTA has seen -- instead of one per warp, which keeps the candidates few
// when a CTA sees only a few hundred kilobytes of a column.
#pragma once

#include "common.cuh"

namespace cta {

constexpr int kWarpsPerCta = 15;                   // streaming warps per CTA
constexpr int kConsumerThreads = kWarpsPerCta * 32;
constexpr int kMergeWarp = kWarpsPerCta;           // folds candidates into the CTA's list, finishes columns
constexpr int kThreads = kConsumerThreads + 32;
constexpr int kLaneVec = 8;                        // 16-byte vectors per lane per chunk
constexpr int kWarpVec = 32 * kLaneVec;            // vectors per warp per chunk (4 KiB)
constexpr int kChunkVec = kWarpsPerCta * kWarpVec; // vectors per chunk (60 KiB)
constexpr int kQuarterWarps = 4;                   // warps fed by one bulk copy (and barrier)
constexpr int kQuarterVec = kQuarterWarps * kWarpVec;
constexpr int kQuarters = (kWarpsPerCta + kQuarterWarps - 1) / kQuarterWarps;
constexpr int kSlots = 3;                          // ring depth (180 KiB per SM)
constexpr int kBufCap = 96;                        // candidate buffer (entries)
constexpr int kSegSlots = 3;                       // segments the streaming warps may run ahead of the merge
constexpr int kMinSliceVec = 1024;                 // smallest slice a CTA is given
constexpr int64_t kSeedElems = 8 * kChunkVec / 2;  // seed a column until the CTA has seen this many elements

static_assert(kBufCap >= SPEC_MAX_K + 32 && kBufCap % 32 == 0, "a pruned buffer must leave room");

// ---- sorted lists -------------------------------------------------------------

// Merge a batch of up to 32 candidates (one per lane; 0 = none) into the
// list lst[0..L) (distinct entries, sorted best first, L <= kk <= 64), keeping
// the kk best; returns the new length.  Every entry's new place is its rank:
// the entries above it in the list plus the candidates above it.
__device__ __forceinline__ int list_merge32(unsigned long long *lst, int L, unsigned long long e, int kk, int lane)
{
    const uint32_t has = __ballot_sync(kFull, e != 0ull);
    if (!has) return L;
    const int b = __popc(has);
    const unsigned long long l0 = lane < L ? lst[lane] : 0ull;
    const unsigned long long l1 = lane + 32 < L ? lst[lane + 32] : 0ull;
    int p0 = lane, p1 = lane + 32, pc = 0;
    if (b <= 8) {
        // few: one pass over the candidates; each one, broadcast, moves the
        // list entries below it down one place; the list entries above it
        // (two ballots) and the candidates above it give its own place
        for (uint32_t mm = has; mm; mm &= mm - 1) {
            const int src = __ffs(mm) - 1;
            const unsigned long long o = __shfl_sync(kFull, e, src);
            pc += o > e;
            p0 += o > l0;
            p1 += o > l1;
            const int above = __popc(__ballot_sync(kFull, l0 > o)) + __popc(__ballot_sync(kFull, l1 > o));
            if (lane == src) pc += above;
        }
    } else {
        // many: sort the batch across the warp (bitonic, best first); a
        // candidate's place is its index plus the list entries above it, a
        // list entry's its index plus the candidates above it (two searches)
#pragma unroll
        for (int k2 = 2; k2 <= 32; k2 <<= 1)
#pragma unroll
            for (int j2 = k2 >> 1; j2 > 0; j2 >>= 1) {
                const unsigned long long o = __shfl_xor_sync(kFull, e, j2);
                const bool first = (lane & j2) == 0, desc = (lane & k2) == 0;
                e = (first == desc) ? (e > o ? e : o) : (e < o ? e : o);
            }
        int lo = 0, hi = L;   // list entries above e
        if (e != 0ull)
            while (lo < hi) {
                const int mid = (lo + hi) >> 1;
                if (lst[mid] > e) lo = mid + 1;
                else hi = mid;
            }
        pc = lane + lo;
        int c0 = 0, c1 = 0;   // batch entries above l0, l1: the first index whose entry is below
#pragma unroll
        for (int step = 16; step >= 1; step >>= 1) {
            const unsigned long long v0 = __shfl_sync(kFull, e, c0 + step - 1);
            const unsigned long long v1 = __shfl_sync(kFull, e, c1 + step - 1);
            if (v0 > l0) c0 += step;
            if (v1 > l1) c1 += step;
        }
        const unsigned long long e31 = __shfl_sync(kFull, e, 31);   // every lane takes part
        if (c0 == 31 && e31 > l0) c0 = 32;
        if (c1 == 31 && e31 > l1) c1 = 32;
        p0 += c0;
        p1 += c1;
    }
    __syncwarp();         // every read of the list is done
    if (lane < L && p0 < kk) lst[p0] = l0;
    if (lane + 32 < L && p1 < kk) lst[p1] = l1;
    if (e != 0ull && pc < kk) lst[pc] = e;
    __syncwarp();
    const int nl = L + b;
    return nl < kk ? nl : kk;
}

// Lane q (< 32) holds the length len of the q-th of up to 32 sources; the
// candidates are numbered source by source.  For candidate g (< total),
// returns its source q and its place in that source.
__device__ __forceinline__ int batch_source(int pre, int g, int &off)
{
    int q = 0;    // the last source starting at or before g
#pragma unroll
    for (int step = 16; step >= 1; step >>= 1) {
        const int cand = q + step;
        const int p = __shfl_sync(kFull, pre, cand < 32 ? cand : 31);
        if (cand < 32 && p <= g) q = cand;
    }
    off = g - __shfl_sync(kFull, pre, q);
    return q;
}

// ---- the per-CTA stream ---------------------------------------------------------

// Shared memory of one CTA: its copy ring, the warps' candidate buffers (two
// slots, rotating by segment), the CTA's list for the current column and
// the copy barriers.
struct CtaSmem {
    uint4 ring[kSlots][kChunkVec];
    unsigned long long wbuf[kWarpsPerCta][kSegSlots][kBufCap];
    unsigned long long cbuf[SPEC_MAX_K];    // the CTA's list for its current column, best first
    unsigned long long tcert;               // ((column + 1) << 16) | certified key of cbuf
    uint64_t full[kSlots][kQuarters];       // a quarter chunk has landed
    uint64_t seg_full[kSegSlots];           // every streaming warp is done with a segment (per slot)
    uint64_t seg_empty[kSegSlots];          // the merging warp is done with a slot
    uint32_t cnt[kSegSlots][kWarpsPerCta];  // entries each warp appended in a segment
    uint32_t done[kSlots];                  // streaming warps done with a slot's chunk
    uint32_t seedmax[2][kWarpsPerCta];
    __align__(16) uint32_t hist[2][2][128]; // seed histograms [parity][pass]: 256 16-bit counts
};

constexpr size_t kSmemBytes = sizeof(CtaSmem);
static_assert(kSmemBytes <= 227 * 1024, "one CTA per SM must fit");
static_assert(kThreads == 512, "four warps per scheduler: up to 128 registers a thread");

// Write a finished column from its sorted list lst[0..n): top-k outputs, or
// for a target column the argmax and, for the lane's last column, the prefix
// match (one lane per position).
__device__ __noinline__ void emit_column(const RoundArgs &a, const Run &r, int64_t c,
                                         const unsigned long long *lst, int n, int lane)
{
    if (r.draft) {
        const int kk = r.kk;
        for (int i = lane; i < n; i += 32) {
            const unsigned long long e = lst[i];
            a.out_vals[c * kk + i] = entry_raw(e);
            a.out_ids[c * kk + i] = (int32_t)entry_id(e);
        }
        return;
    }
    if (a.uniforms) sampled_column_done(a, c, lst, n, lane);
    else verify_column_done(a, c, n > 0 ? (int32_t)entry_id(lst[0]) : 0, lane);
}

// Column c's part in slice w is over and its best entries are the sorted
// list lst[0..n).  If the slice holds the whole column, emit it; otherwise
// publish the list and take the column's ticket; the slice that completes the
// column merges every slice's list and emits the result.  Returns 0 (the
// CTA's list is free again).
__device__ __noinline__ int finish_column(const RoundArgs &a, const Run &r, int w, int64_t c,
                                          unsigned long long *lst, int n, int lane)
{
    const int kk = r.kk;
    const int64_t wf = owner(r, (c * r.V + r.mis) >> 3);
    const int64_t wl = owner(r, ((c + 1) * r.V - 1 + r.mis) >> 3);
    if (wf == wl) {
        emit_column(a, r, c, lst, n, lane);
        return 0;
    }
    // publish: the list, then its length in slot kk
    unsigned long long *mine = list_slot(a, r, w, c);
    for (int i = lane; i < n; i += 32) mine[i] = lst[i];
    if (lane == 0) mine[kk] = (unsigned long long)n;
    __syncwarp();
    // the ticket: release (the list above is visible first) and acquire
    // (every earlier list is visible to the last) in one atomic
    const int64_t tix = r.draft ? c : a.d_cols + c;
    unsigned last = 0;
    if (lane == 0) last = atom_add_acq_rel(a.col_ticket + tix, 1u) == (unsigned)(wl - wf);
    if (!__shfl_sync(kFull, last, 0)) return 0;
    __syncwarp();
    // merge every slice's list.  The best certificate of a full list (its
    // kk-th key) bounds the column's kk-th key: entries below it are left
    // out.
    n = 0;
    const int64_t nparts = wl - wf + 1;
    if (nparts <= 32 && nparts * kk <= 128) {
        // few short lists: lengths, certificates and every list slot in one
        // round of loads, four slots a lane
        const unsigned long long *mylist = lane < nparts ? list_slot(a, r, wf + lane, c) : nullptr;
        const int len = mylist ? (int)__ldcg(mylist + kk) : 0;
        const unsigned long long lastv = mylist ? __ldcg(mylist + kk - 1) : 0ull;
        unsigned long long ent[4];
        int slot[4], from[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int g = lane + 32 * i;
            from[i] = g < nparts * kk ? g / kk : 0;
            slot[i] = g - from[i] * kk;
            const unsigned long long *src = reinterpret_cast<const unsigned long long *>(
                __shfl_sync(kFull, reinterpret_cast<uintptr_t>(mylist), from[i]));
            ent[i] = g < nparts * kk ? __ldcg(src + slot[i]) : 0ull;
        }
        const uint32_t cert = __reduce_max_sync(kFull, len == kk ? entry_key(lastv) : 0u);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int lq = __shfl_sync(kFull, len, from[i]);
            unsigned long long e = slot[i] < lq ? ent[i] : 0ull;   // slots past a list's length are stale
            if (entry_key(e) < cert || (n == kk && e < lst[kk - 1])) e = 0ull;
            n = list_merge32(lst, n, e, kk, lane);
        }
        emit_column(a, r, c, lst, n, lane);
        if (lane == 0) a.col_ticket[tix] = 0u;   // ready for the next launch
        return 0;
    }
    for (int64_t q0 = 0; q0 < nparts; q0 += 32) {
        const unsigned long long *mylist = q0 + lane < nparts ? list_slot(a, r, wf + q0 + lane, c) : nullptr;
        const int len = mylist ? (int)__ldcg(mylist + kk) : 0;
        const unsigned long long last = mylist ? __ldcg(mylist + kk - 1) : 0ull;
        const uint32_t cert = __reduce_max_sync(kFull, len == kk ? entry_key(last) : 0u);
        int total;
        const int pre = warp_exclusive_sum(len, lane, total);
        for (int base = 0; base < total; base += 32) {
            int off;
            const int q = batch_source(pre, base + lane, off);
            const unsigned long long *src = reinterpret_cast<const unsigned long long *>(
                __shfl_sync(kFull, reinterpret_cast<uintptr_t>(mylist), q));
            unsigned long long e = base + lane < total ? __ldcg(src + off) : 0ull;
            if (entry_key(e) < cert || (n == kk && e < lst[kk - 1])) e = 0ull;
            n = list_merge32(lst, n, e, kk, lane);
        }
    }
    emit_column(a, r, c, lst, n, lane);
    if (lane == 0) a.col_ticket[tix] = 0u;   // ready for the next launch
    return 0;
}

// Issue the bulk copies of chunk i of slice [J0, J1) into ring slot
// i % kSlots, one per quarter (each completing on its own barrier).  Only
// vectors wholly inside the buffer are copied; the (at most two) edge vectors
// of the buffer are read element by element by the consumer.
__device__ __forceinline__ void issue_chunk(const Run &r, CtaSmem &s, int64_t J0, int64_t J1, int64_t i)
{
    const int sl = (int)(i % kSlots);
    const int64_t vs = J0 + i * kChunkVec;
    const int64_t ve = vs + kChunkVec < J1 ? vs + kChunkVec : J1;
    fence_proxy_async();
#pragma unroll 1
    for (int q = 0; q < kQuarters; ++q) {
        const int64_t qs = vs + (int64_t)q * kQuarterVec;
        const int64_t qe = qs + kQuarterVec < ve ? qs + kQuarterVec : ve;
        const int64_t is = qs > r.jlo ? qs : r.jlo;
        const int64_t ie = qe < r.jhi ? qe : r.jhi;
        const uint32_t bytes = ie > is ? (uint32_t)((ie - is) * 16) : 0u;
        mbar_arrive_expect_tx(&s.full[sl][q], bytes);
        if (bytes) bulk_g2s(&s.ring[sl][is - vs], r.vb + is, bytes, &s.full[sl][q]);
    }
}

// ---- consumer-only barrier (named barrier 1: the 16 streaming warps) ----------

__device__ __forceinline__ void consumers_sync() { asm volatile("bar.sync 1, %0;" ::"n"(kConsumerThreads) : "memory"); }

__device__ __forceinline__ void mbar_arrive(uint64_t *bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// Histogram h (256 bins of 16-bit counts, two per word, lane l holding bins
// 8l..8l+7): find the bin b where the count from the top first reaches
// need; on return need is what is still wanted inside b.  False if the
// whole histogram holds fewer than need.
__device__ __forceinline__ bool select_bin(const uint32_t *h, int &need, int lane, int &bin)
{
    const uint4 q = reinterpret_cast<const uint4 *>(h)[lane];
    const uint32_t wd[4] = {q.x, q.y, q.z, q.w};
    int tot = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) tot += (int)(wd[i] & 0xFFFFu) + (int)(wd[i] >> 16);
    int suf = tot;   // bins of this lane and every higher lane
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const int y = __shfl_down_sync(kFull, suf, d);
        if (lane + d < 32) suf += y;
    }
    const uint32_t ok = __ballot_sync(kFull, suf >= need);
    if (!ok) return false;
    const int L = 31 - __clz((int)ok);
    int b = 0, rem = 0, above = suf - tot;
    bool found = false;
#pragma unroll
    for (int e = 7; e >= 0; --e) {
        const int ce = (int)((wd[e >> 1] >> (16 * (e & 1))) & 0xFFFFu);
        if (!found && above + ce >= need) {
            found = true;
            b = 8 * lane + e;
            rem = need - above;
        }
        above += ce;
    }
    bin = __shfl_sync(kFull, b, L);
    need = __shfl_sync(kFull, rem, L);
    return true;
}

// Count key into histogram h at bin (warp-aggregated shared-memory atomics).
__device__ __forceinline__ void hist_add(uint32_t *h, bool in, uint32_t bin, int lane)
{
    const uint32_t peers = __match_any_sync(kFull, in ? bin : 0xFFFFFFFFu);
    if (in && lane == __ffs(peers) - 1) atomicAdd(&h[bin >> 1], (uint32_t)__popc(peers) << (16 * (bin & 1)));
}

// The kk-th largest of the streaming warps' per-thread keys (0 if fewer than
// kk are non-zero): two passes of a 256-bin histogram, on the high and then
// the low byte of the keys; for kk = 1 a plain maximum.  Every streaming
// thread must call it, with `par` alternating between calls: the histograms
// and maxima are double buffered (the streaming warps stay within one call
// of each other), and each call clears the other parity's histograms.
__device__ __forceinline__ uint32_t seed_kth(uint32_t key, int kk, CtaSmem &s, int lane, int w, int par)
{
    if (kk == 1) {
        const uint32_t m = __reduce_max_sync(kFull, key);
        if (lane == 0) s.seedmax[par][w] = m;
        consumers_sync();
        const uint32_t t = lane < kWarpsPerCta ? s.seedmax[par][lane] : 0u;
        return __reduce_max_sync(kFull, t);
    }
    uint32_t *h1 = s.hist[par][0], *h2 = s.hist[par][1];
    hist_add(h1, key != 0, key >> 8, lane);
    consumers_sync();
    // every warp has read the previous call's histograms before this barrier
    constexpr int kClr = (256 + kWarpsPerCta - 1) / kWarpsPerCta;   // words each warp clears
    if (lane < kClr && w * kClr + lane < 256) {
        const int idx = w * kClr + lane;
        s.hist[par ^ 1][idx >> 7][idx & 127] = 0u;
    }
    int need = kk, b1 = 0, b2 = 0;
    if (!select_bin(h1, need, lane, b1)) {
        consumers_sync();   // keep the barrier sequence the same in every warp
        return 0;
    }
    hist_add(h2, key != 0 && (int)(key >> 8) == b1, key & 0xFFu, lane);
    consumers_sync();
    select_bin(h2, need, lane, b2);
    return ((uint32_t)b1 << 8) | (uint32_t)b2;
}

// Fold every streaming warp's candidates of a segment (slot h of the warp
// buffers) into the CTA's sorted list lst[0..n) for column c; publish the
// list's certificate (the key of its kk-th entry).  Returns the new length.
__device__ __forceinline__ int merge_segment(const Run &r, int64_t c, CtaSmem &s, int h, int n, int lane)
{
    const int kk = r.kk;
    uint32_t cw[kWarpsPerCta];
    int total = 0;
#pragma unroll
    for (int q = 0; q < kWarpsPerCta; ++q) {
        cw[q] = s.cnt[h][q];
        total += (int)cw[q];
    }
    if (total == 0) return n;
    for (int base = 0; base < total; base += 32) {
        // candidate g = base + lane: find its warp by scanning the counts
        const int g = base + lane;
        int acc = 0, q = -1, off = 0;
#pragma unroll
        for (int w2 = 0; w2 < kWarpsPerCta; ++w2) {
            if (q < 0 && g < acc + (int)cw[w2]) {
                q = w2;
                off = g - acc;
            }
            acc += (int)cw[w2];
        }
        unsigned long long e = q >= 0 ? s.wbuf[q][h][off] : 0ull;
        if (n == kk && e < s.cbuf[kk - 1]) e = 0ull;   // below a full list's kk-th: cannot enter
        n = list_merge32(s.cbuf, n, e, kk, lane);
    }
    if (n == kk && lane == 0)
        *reinterpret_cast<volatile unsigned long long *>(&s.tcert) =
            ((unsigned long long)(c + 1) << 16) | entry_key(s.cbuf[kk - 1]);
    return n;
}

// The segments of a slice: chunk i covers vectors [vs, ve) and elements
// [g_first, g_end) of the run; the part of column c inside it is a segment.
// The streaming warps and the merging warp walk the same sequence.
struct Chunk {
    int64_t vs, ve, g_first, g_end;
};

__device__ __forceinline__ Chunk chunk_of(const Run &r, int64_t J0, int64_t J1, int64_t i)
{
    Chunk k;
    k.vs = J0 + i * kChunkVec;
    k.ve = k.vs + kChunkVec < J1 ? k.vs + kChunkVec : J1;
    k.g_first = 8 * k.vs - r.mis > 0 ? 8 * k.vs - r.mis : 0;
    k.g_end = 8 * k.ve - r.mis < r.N ? 8 * k.ve - r.mis : r.N;   // exclusive
    return k;
}

// The merging warp: it folds each segment's candidates into the CTA's list
// as soon as the streaming warps are done with it, frees the segment's
// buffers, and finishes columns.
__device__ __noinline__ void merge_slice(const RoundArgs &a, const Run &r, int64_t J0, int64_t J1, int bi,
                                         CtaSmem &s, int lane)
{
    const int64_t nch = (J1 - J0 + kChunkVec - 1) / kChunkVec;
    int64_t c = udiv(first_elem(r, bi), r.V);
    int sg = 0, n = 0;
    for (int64_t i = 0; i < nch; ++i) {
        const Chunk k = chunk_of(r, J0, J1, i);
        for (;;) {
            const int64_t ce = (c + 1) * r.V;
            const bool col_ends = ce <= k.g_end;
            const int h = sg % kSegSlots;
            mbar_wait(&s.seg_full[h], (uint32_t)(sg / kSegSlots) & 1u);
            n = merge_segment(r, c, s, h, n, lane);
            __syncwarp();
            if (lane == 0) mbar_arrive(&s.seg_empty[h]);
            if (col_ends || i + 1 == nch) n = finish_column(a, r, bi, c, s.cbuf, n, lane);
            ++sg;
            if (!col_ends) break;                         // column c goes on past this chunk
            ++c;
            if (c * r.V >= k.g_end) break;                // next column starts in a later chunk
        }
    }
}

// A warp's share of a chunk restricted to column [cb, ce), elements outside
// it as NaN (the general case: a column or buffer edge inside the share, or
// a partial chunk).  The buffer's edge vectors, which the bulk copies leave
// out, are read here and stored into the ring, masked to the column.
__device__ __forceinline__ void load_share_masked(const Run &r, CtaSmem &s, int sl, int64_t vs, int64_t wvs,
                                                  int64_t wve, int64_t cb, int64_t ce, int lane,
                                                  uint4 (&y)[kLaneVec])
{
#pragma unroll
    for (int u = 0; u < kLaneVec; ++u) {
        const int64_t j = wvs + u * 32 + lane;
        if (j >= wve) {
            y[u] = make_uint4(kNaN2, kNaN2, kNaN2, kNaN2);
            continue;
        }
        uint4 q;
        if (j < r.jlo || j >= r.jhi) {
            q = load_edge(r.buf, j, r.mis, cb, ce < r.N ? ce : r.N);
            s.ring[sl][j - vs] = q;
            fence_proxy_async();
        } else {
            q = s.ring[sl][j - vs];
        }
        const int64_t g0 = 8 * j - r.mis;
        uint32_t wv[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
        for (int hh = 0; hh < 4; ++hh) {
            const int64_t ga = g0 + 2 * hh;
            if (ga < cb || ga >= ce) wv[hh] = (wv[hh] & 0xFFFF0000u) | 0x7FFFu;
            if (ga + 1 < cb || ga + 1 >= ce) wv[hh] = (wv[hh] & 0x0000FFFFu) | 0x7FFF0000u;
        }
        y[u] = make_uint4(wv[0], wv[1], wv[2], wv[3]);
    }
}

// Append the candidates of a warp's share y (elements that pass f; masked
// elements are NaN and never pass) to the warp buffer wb; returns its new
// length.  One warp prefix sum gives every lane its places; their order in
// the buffer does not matter.  Values are read back from the ring (the
// share's own bits).  A full buffer is pruned to its kk best, and what is
// left of the share is then filtered (inclusively) against their
// certificate.
__device__ __forceinline__ int append_share(const Run &r, const uint4 (&y)[kLaneVec], const uint16_t *sv,
                                            int64_t id_lane, const Filter f, const int32_t *__restrict__ id_map,
                                            unsigned long long *wb, int lane)
{
    const int kk = r.kk;
    uint64_t bits = 0;   // this lane's candidates: bit 8u+e = element e of vector u
#pragma unroll
    for (int u = 0; u < kLaneVec; ++u)
        if (f.strict ? any_gt(vmax(y[u]), f.thr2) : any_ge(vmax(y[u]), f.thr2))
            bits |= (uint64_t)elem_mask(y[u], f) << (8 * u);
    int n = 0;
    for (;;) {
        int total;
        const int excl = warp_exclusive_sum(__popcll(bits), lane, total);
        if (total == 0) break;
        const int space = kBufCap - n;
        int pos = excl;
        uint64_t rest = bits;
        while (rest && pos < space) {
            const int b = __ffsll((long long)rest) - 1;
            rest &= rest - 1;
            const int u = b >> 3, e = b & 7;
            uint32_t cid = (uint32_t)(id_lane + 256 * u + e);
            if (id_map) cid = (uint32_t)__ldg(id_map + cid);
            wb[n + pos] = pack_entry(bf16_as_float(sv[8 * (u * 32 + lane) + e]), cid);
            ++pos;
        }
        __syncwarp();
        if (total <= space) {
            n += total;
            break;
        }
        const Pruned pq = buf_prune<kBufCap / 32>(wb, kBufCap, kk, lane);
        n = pq.n;
        const float tv = bf16_as_float(key_to_raw(pq.t));
        uint64_t keep = 0;
        for (uint64_t q = rest; q; q &= q - 1) {
            const int b = __ffsll((long long)q) - 1;
            if (bf16_as_float(sv[8 * ((b >> 3) * 32 + lane) + (b & 7)]) >= tv) keep |= 1ull << b;
        }
        bits = keep;
    }
    return n;
}

// A streaming warp w of slice bi takes vectors [w * kWarpVec, (w + 1) *
// kWarpVec) of every chunk.  Per segment it filters its share against the
// column's certificate and appends its candidates to buffer slot sg % kSegSlots,
// then hands the slot to the merging warp.  id_map is null for token ids.
__device__ __forceinline__ void stream_slice(const RoundArgs &a, const Run &r, int bi, int64_t J0, int64_t J1,
                                             const int32_t *__restrict__ id_map, CtaSmem &s, int lane, int w)
{
    const int64_t nch = (J1 - J0 + kChunkVec - 1) / kChunkVec;
    const int kk = r.kk;
    int64_t c = udiv(first_elem(r, bi), r.V);       // current column
    int64_t seen = 0;                          // elements of column c this CTA has scanned
    uint32_t tprev = 0;                        // best seed of column c from an earlier chunk
    int sg = 0, nseed = 0;

    for (int64_t i = 0; i < nch; ++i) {
        const int sl = (int)(i % kSlots);
        mbar_wait(&s.full[sl][w / kQuarterWarps], (uint32_t)(i / kSlots) & 1u);
        const Chunk k = chunk_of(r, J0, J1, i);
        const int64_t wvs = k.vs + (int64_t)w * kWarpVec;                        // this warp's vectors
        const int64_t wve = wvs + kWarpVec < k.ve ? wvs + kWarpVec : k.ve;
        for (;;) {
            const int64_t cb = c * r.V, ce = cb + r.V;
            // the warp's share of column c, elements outside it as NaN
            uint4 y[kLaneVec];
            if (wve > wvs && 8 * wve - r.mis > cb && 8 * wvs - r.mis < ce) {
                if (wve - wvs == kWarpVec && wvs >= r.jlo && wve <= r.jhi && cb <= 8 * wvs - r.mis &&
                    ce >= 8 * wve - r.mis) {
                    // the common case: a full share, inside one column, no buffer edge
                    const uint4 *src = &s.ring[sl][wvs - k.vs + lane];
#pragma unroll
                    for (int u = 0; u < kLaneVec; ++u) y[u] = src[u * 32];
                } else {
                    load_share_masked(r, s, sl, k.vs, wvs, wve, cb, ce, lane, y);
                }
            } else {
#pragma unroll
                for (int u = 0; u < kLaneVec; ++u) y[u] = make_uint4(kNaN2, kNaN2, kNaN2, kNaN2);
            }
            uint32_t m = vmax(y[0]);
#pragma unroll
            for (int u = 1; u < kLaneVec; ++u) m = bmax2(m, vmax(y[u]));

            // seed, until the CTA has scanned a good part of the column: the
            // kk-th largest of the 512 lane maxima (groups of 64 elements)
            // certifies kk elements; the decision is the same in every warp
            uint32_t tseed = 0;
            if (seen < kSeedElems) tseed = seed_kth(order_key(hmax_splat(m) & 0xFFFFu), kk, s, lane, w, nseed++ & 1);
            // the CTA list's certificate lags (its merge runs while the warps
            // filter the next segments); seeds of earlier chunks stand in
            // meanwhile.  Both are certified by elements of earlier chunks, so
            // they filter strictly (token ids); this chunk's seed inclusively.
            const unsigned long long tc = *reinterpret_cast<volatile unsigned long long *>(&s.tcert);
            uint32_t tcta = (tc >> 16) == (unsigned long long)(c + 1) ? (uint32_t)(tc & 0xFFFFu) : 0u;
            tcta = tprev > tcta ? tprev : tcta;
            const Filter f = make_filter(tcta, tseed, id_map != nullptr);

            const int h = sg % kSegSlots;
            // buffer slot h is free once the merge of segment sg - kSegSlots is done
            if (sg >= kSegSlots) mbar_wait(&s.seg_empty[h], (uint32_t)((sg - kSegSlots) / kSegSlots) & 1u);
            int n = 0;
            if (__ballot_sync(kFull, f.strict ? any_gt(m, f.thr2) : any_ge(m, f.thr2)))
                n = append_share(r, y, reinterpret_cast<const uint16_t *>(&s.ring[sl][wvs - k.vs]),
                                 8 * (wvs + lane) - r.mis - cb, f, id_map, s.wbuf[w][h], lane);
            if (lane == 0) s.cnt[h][w] = (uint32_t)n;
            __syncwarp();
            if (lane == 0) mbar_arrive(&s.seg_full[h]);   // the segment's share is in

            ++sg;
            const int64_t lo = cb > k.g_first ? cb : k.g_first, hi = ce < k.g_end ? ce : k.g_end;
            seen += hi - lo;
            tprev = tseed > tprev ? tseed : tprev;
            if (ce > k.g_end) break;                      // column c goes on past this chunk
            ++c;
            seen = 0;
            tprev = 0;
            if (c * r.V >= k.g_end) break;                // next column starts in a later chunk
        }
        // the warp is done with slot sl: the last warp to get here refills
        // it with chunk i + kSlots
        __syncwarp();
        if (lane == 0) {
            __threadfence_block();   // the warp's reads of the slot come first
            if (atomicAdd(&s.done[sl], 1u) == kWarpsPerCta - 1) {
                __threadfence_block();
                s.done[sl] = 0u;
                if (i + kSlots < nch) issue_chunk(r, s, J0, J1, i + kSlots);
            }
        }
    }
}

__global__ void __launch_bounds__(kThreads, 1) spec_round_kernel(const __grid_constant__ RoundArgs a)
{
    pdl_launch_dependents();
    pdl_wait();
    extern __shared__ __align__(128) unsigned char smem[];
    CtaSmem &s = *reinterpret_cast<CtaSmem *>(smem);
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const int b = blockIdx.x;
    if (b >= a.d_units + a.t_units) return;

    Run r;
    const bool draft = b < a.d_units;
    r.draft = draft;
    r.buf = draft ? a.draft : a.target;
    r.V = draft ? a.d_V : a.t_V;
    r.N = (draft ? a.d_cols : a.t_cols) * r.V;
    r.W = draft ? a.d_units : a.t_units;
    r.gw0 = draft ? 0 : a.d_units;
    r.kk = draft ? a.k : a.t_k;
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(r.buf);
    r.mis = (int)((a0 >> 1) & 7);                       // element phase of buf in 16 B
    r.vb = reinterpret_cast<const uint4 *>(a0 - 2 * (uintptr_t)r.mis);
    r.NV = (r.N + r.mis + 7) >> 3;
    r.jlo = r.mis ? 1 : 0;
    r.jhi = ((r.N + r.mis) & 7) ? r.NV - 1 : r.NV;
    if (r.jhi < r.jlo) r.jhi = r.jlo;
    const int bi = b - r.gw0;
    const int64_t J0 = slice_start(r, bi), J1 = slice_start(r, bi + 1);
    if (J1 <= J0) return;

    if (threadIdx.x == 0) {
        for (int sl = 0; sl < kSlots; ++sl)
            for (int q = 0; q < kQuarters; ++q) mbar_init(&s.full[sl][q], 1);
        for (int h = 0; h < kSegSlots; ++h) {
            mbar_init(&s.seg_full[h], kWarpsPerCta);
            mbar_init(&s.seg_empty[h], 1);
        }
        fence_mbar_init();
        s.tcert = 0ull;
        s_gave_up = 0u;
        for (int sl = 0; sl < kSlots; ++sl) s.done[sl] = 0u;
        const int64_t nch = (J1 - J0 + kChunkVec - 1) / kChunkVec;
        for (int64_t i = 0; i < nch && i < kSlots; ++i) issue_chunk(r, s, J0, J1, i);
    }
    for (int i = threadIdx.x; i < 2 * 2 * 128; i += kThreads) (&s.hist[0][0][0])[i] = 0u;
    __syncthreads();
    if (w == kMergeWarp) merge_slice(a, r, J0, J1, bi, s, lane);
    else stream_slice(a, r, bi, J0, J1, draft ? a.id_map : nullptr, s, lane, w);
}

}  // namespace cta
