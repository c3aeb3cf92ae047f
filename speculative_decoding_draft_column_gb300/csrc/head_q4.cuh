// The Q4 shortlist head ("A drafter inside the artifact", Ignis DFlash2 page,
// section "How it works", second paragraph: an opt-in 4-bit head over the
// 131,072 most frequent tokens, about 356 MB): logits of every head row for
// a few hidden states, on the tensor cores.
//
// Layout of the head as callers hold it: weights uint8 [rows][d/2], byte j of
// a row holding weight 2j in its low nibble and 2j+1 in its high nibble, a
// nibble n standing for n - 8; fp16 scales [rows][d/64], one per block of 64
// weights.  A logit is sum_b scale_b * sum_{j in block b} (n_j - 8) * h_j.
//
// pack_kernel reorders that, once, into tiles of 16 rows x 64 weights in the
// order of the mma.sync m16n8k16 A fragment, so that each lane of a warp
// loads one 16-byte word per tile and block (coalesced, 512 B a warp) and
// turns two nibbles into a bf16 pair with one lop3 and one subtraction:
// bf16 0x4300 | n is 128 + n, and 128 + n - 136 = n - 8 exactly.  The
// block's products are summed by the tensor cores in fp32 (each k16 step from
// zero into an accumulator of its own, so that the four MMAs of a block do not
// wait on each other, then the four added), and the block's per-row scale is
// applied in registers (one FMA per accumulator), so every 64-weight partial
// sum gets its own scale.  A TMEM accumulator
// (tcgen05) would need a TMEM round trip per block and tile for that, which
// is why this contraction stays on the register-accumulator MMA.
#pragma once

#include "common.cuh"

namespace q4 {

constexpr int kWarps = 16;
constexpr int kThreads = kWarps * 32;
constexpr int kNT = 2;                    // n-tiles of 8 hidden states per pass
constexpr int kColsPass = 8 * kNT;        // hidden states per pass over the head
constexpr int kAhead = 8;                 // blocks of weights a lane loads together
constexpr int kPadWords = 4;              // padding of a staged hidden state (spreads the banks)
constexpr int64_t kMaxD = 6144;           // staged hidden states must fit in shared memory

// staged hidden states (bf16 pairs, padded rows)
inline size_t smem_bytes(int64_t d, int nt) { return (size_t)(8 * nt) * (size_t)(d / 2 + kPadWords) * 4; }

// One packed word: tile T, block B, lane L = 4g + t, k16 step s holds the
// nibbles of (row 16T+g / 16T+g+8, weight 64B + 16s + 2t + {0, 1, 8, 9}) at
// bits  0-3: (g, +0)   16-19: (g, +1)    4-7: (g+8, +0)   20-23: (g+8, +1)
//       8-11: (g, +8)  24-27: (g, +9)   12-15: (g+8, +8)  28-31: (g+8, +9)
// so that (word >> 4r) & 0x000F000F is the nibble pair of A register r.
// Scale word [T][B][g] = scale(row 16T+g) | scale(row 16T+g+8) << 16.
__global__ void pack_kernel(const uint8_t *__restrict__ wq, const uint16_t *__restrict__ sc, int64_t rows, int64_t d,
                            uint32_t *__restrict__ wp, uint32_t *__restrict__ sp)
{
    const int64_t nb = d / 64, total = rows / 16 * nb * 128;
    const int64_t half = d / 2;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
        const int s = (int)(i & 3), L = (int)((i >> 2) & 31);
        const int64_t tb = i >> 7, B = tb % nb, T = tb / nb;
        const int g = L >> 2, t = L & 3;
        const int64_t r0 = T * 16 + g, r1 = r0 + 8, k0 = B * 64 + 16 * s + 2 * t;
        const uint8_t *p0 = wq + r0 * half, *p1 = wq + r1 * half;
        // k0 is even: weights k0, k0+1 share byte k0/2 (low, high nibble), and so do k0+8, k0+9
        const uint32_t b00 = p0[k0 / 2], b01 = p0[k0 / 2 + 4], b10 = p1[k0 / 2], b11 = p1[k0 / 2 + 4];
        wp[i] = (b00 & 0xFu) | ((b00 >> 4) << 16) | ((b10 & 0xFu) << 4) | ((b10 >> 4) << 20) | ((b01 & 0xFu) << 8) |
                ((b01 >> 4) << 24) | ((b11 & 0xFu) << 12) | ((b11 >> 4) << 28);
        if (s == 0 && t == 0) sp[tb * 8 + g] = (uint32_t)sc[r0 * nb + B] | ((uint32_t)sc[r1 * nb + B] << 16);
    }
}

__device__ __forceinline__ uint32_t lop3_and_or(uint32_t a, uint32_t b, uint32_t c)
{
    uint32_t d;
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "r"(b), "r"(c));   // (a & b) | c
    return d;
}

__device__ __forceinline__ uint32_t sub_bf16x2(uint32_t a, uint32_t b)
{
    uint32_t d;
    asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// fp32 -> bf16 bit pattern, to nearest, ties to even (the hardware conversion)
__device__ __forceinline__ uint16_t bf16_rn(float f)
{
    uint16_t h;
    asm("{\n\t.reg .b16 r;\n\tcvt.rn.bf16.f32 r, %1;\n\tmov.b16 %0, r;\n\t}" : "=h"(h) : "f"(f));
    return h;
}

__device__ __forceinline__ float f16_as_float(uint32_t bits16)
{
    float f;
    asm("{\n\t.reg .f16 h;\n\tmov.b16 h, %1;\n\tcvt.f32.f16 %0, h;\n\t}" : "=f"(f) : "h"((unsigned short)bits16));
    return f;
}

// D = A B (+ 0): m16n8k16, A row-major bf16 (4 registers), B col-major bf16
// (2 registers), D fp32.
__device__ __forceinline__ void mma_bf16(float (&dd)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1, bool zero)
{
    const float c0 = zero ? 0.f : dd[0], c1 = zero ? 0.f : dd[1], c2 = zero ? 0.f : dd[2], c3 = zero ? 0.f : dd[3];
    asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
                 "{%10,%11,%12,%13};"
                 : "=f"(dd[0]), "=f"(dd[1]), "=f"(dd[2]), "=f"(dd[3])
                 : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(c0), "f"(c1), "f"(c2), "f"(c3));
}

__device__ __forceinline__ void cp_async16(void *smem_dst, const void *gmem_src)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(smem_dst)), "l"(gmem_src) : "memory");
}

// Logits of hidden states c0 .. c0 + 8*NT - 1 (fewer at the end) for every
// row of the packed head: logits[c][row] (bf16, round to nearest even from
// the fp32 sum).  Each warp takes whole tiles of 16 rows.
//
// The weights enter the MMA as their exact values n - 8 (bf16 0x4300 | n is
// 128 + n; minus 136 exactly): folding the offset out of the sum instead
// would make every block's sum about 30 times larger than its terms, and its
// rounding with it.
template <int NT>
__global__ void __launch_bounds__(kThreads, 1)
    logits_kernel(const uint16_t *__restrict__ hidden, int64_t cols, int64_t d, const uint4 *__restrict__ wp,
                  const uint32_t *__restrict__ sp, int64_t rows, int64_t c0, uint16_t *__restrict__ logits)
{
    pdl_launch_dependents();
    pdl_wait();
    extern __shared__ uint32_t hs[];   // [8*NT][d/2 + kPadWords] bf16 pairs
    const int words = (int)(d / 2), stride = words + kPadWords, nb = (int)(d / 64);
    const int nc = (int)(cols - c0 < 8 * NT ? cols - c0 : 8 * NT);
    {
        const int q4w = words / 4;   // 16-byte pieces of a hidden state
        const uint4 *src = reinterpret_cast<const uint4 *>(hidden + c0 * d);
        for (int i = threadIdx.x; i < 8 * NT * q4w; i += kThreads) {
            const int c = i / q4w, j = i - c * q4w;
            uint4 *dst = reinterpret_cast<uint4 *>(hs + c * stride) + j;
            if (c < nc) cp_async16(dst, src + (int64_t)c * q4w + j);
            else *dst = make_uint4(0, 0, 0, 0);
        }
        asm volatile("cp.async.wait_all;" ::: "memory");
        __syncthreads();
    }

    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5, g = lane >> 2, t = lane & 3;
    const int64_t tiles = rows / 16;
    const int64_t nwarps = (int64_t)gridDim.x * kWarps;
    const uint32_t kMask = 0x000F000Fu, kBias = 0x43004300u, kOff = 0x43084308u;   // 128 + n; 136 = 128 + 8
    const uint32_t *hrow[NT];
#pragma unroll
    for (int n = 0; n < NT; ++n) hrow[n] = hs + (n * 8 + g) * stride + t;

    for (int64_t T = (int64_t)blockIdx.x * kWarps + w; T < tiles; T += nwarps) {
        const uint4 *wt = wp + T * nb * 32 + lane;
        const uint32_t *st = sp + T * nb * 8 + g;
        float acc[NT][4];
#pragma unroll
        for (int n = 0; n < NT; ++n) acc[n][0] = acc[n][1] = acc[n][2] = acc[n][3] = 0.f;
        // kAhead blocks of the tile at a time, double buffered: the next
        // group's loads all go out together before this group's arithmetic
        // (issued as a group the loads stay in flight together; refilling one
        // slot per block as it is used held the stream to about a third of
        // the rate)
        auto load_group = [&](int B0, uint4 (&pw)[kAhead], uint32_t (&ps)[kAhead]) {
#pragma unroll
            for (int a = 0; a < kAhead; ++a) {
                const bool in = B0 + a < nb;
                pw[a] = in ? __ldcs(wt + (B0 + a) * 32) : make_uint4(0, 0, 0, 0);
                ps[a] = in ? __ldg(st + (B0 + a) * 8) : 0u;
            }
        };
        auto run_group = [&](int B0, const uint4 (&pw)[kAhead], const uint32_t (&ps)[kAhead]) {
#pragma unroll
            for (int a = 0; a < kAhead; ++a) {
                const int B = B0 + a;
                if (B < nb) {
                    const uint4 wv = pw[a];
                    const uint32_t sv = ps[a];
                    float dd[NT][4];
                    const uint32_t wds[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
                    for (int s = 0; s < 4; ++s) {
                        const uint32_t word = wds[s];
                        const uint32_t ar[4] = {sub_bf16x2(lop3_and_or(word, kMask, kBias), kOff),
                                                sub_bf16x2(lop3_and_or(word >> 4, kMask, kBias), kOff),
                                                sub_bf16x2(lop3_and_or(word >> 8, kMask, kBias), kOff),
                                                sub_bf16x2(lop3_and_or(word >> 12, kMask, kBias), kOff)};
                        const int kw = B * 32 + 8 * s;   // word offset of k in a staged row
#pragma unroll
                        for (int n = 0; n < NT; ++n) mma_bf16(dd[n], ar, hrow[n][kw], hrow[n][kw + 4], s == 0);
                    }
                    const float s0 = f16_as_float(sv & 0xFFFFu), s1 = f16_as_float(sv >> 16);
#pragma unroll
                    for (int n = 0; n < NT; ++n) {
                        acc[n][0] = fmaf(s0, dd[n][0], acc[n][0]);
                        acc[n][1] = fmaf(s0, dd[n][1], acc[n][1]);
                        acc[n][2] = fmaf(s1, dd[n][2], acc[n][2]);
                        acc[n][3] = fmaf(s1, dd[n][3], acc[n][3]);
                    }
                }
            }
        };
        uint4 pa[kAhead], pb[kAhead];
        uint32_t sa[kAhead], sb[kAhead];
        load_group(0, pa, sa);
        for (int B0 = 0; B0 < nb; B0 += 2 * kAhead) {
            if (B0 + kAhead < nb) load_group(B0 + kAhead, pb, sb);
            run_group(B0, pa, sa);
            if (B0 + kAhead >= nb) break;
            if (B0 + 2 * kAhead < nb) load_group(B0 + 2 * kAhead, pa, sa);
            run_group(B0 + kAhead, pb, sb);
        }
        const int64_t r0 = T * 16 + g, r1 = r0 + 8;
#pragma unroll
        for (int n = 0; n < NT; ++n) {
            const int cc = n * 8 + 2 * t;
            if (cc < nc) {
                logits[(c0 + cc) * rows + r0] = bf16_rn(acc[n][0]);
                logits[(c0 + cc) * rows + r1] = bf16_rn(acc[n][2]);
            }
            if (cc + 1 < nc) {
                logits[(c0 + cc + 1) * rows + r0] = bf16_rn(acc[n][1]);
                logits[(c0 + cc + 1) * rows + r1] = bf16_rn(acc[n][3]);
            }
        }
    }
}

}  // namespace q4
