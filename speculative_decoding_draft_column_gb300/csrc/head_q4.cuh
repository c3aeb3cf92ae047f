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
// block's products are summed by the tensor cores in fp32 from zero, and the
// block's per-row scale is applied in registers (one FMA per accumulator), so
// every 64-weight partial sum gets its own scale.  A TMEM accumulator
// (tcgen05) would need a TMEM round trip per block and tile for that, which
// is why this contraction stays on the register-accumulator MMA.
#pragma once

#include "common.cuh"

namespace q4 {

constexpr int kWarps = 16;
constexpr int kThreads = kWarps * 32;
constexpr int kNT = 2;                    // n-tiles of 8 hidden states per pass
constexpr int kColsPass = 8 * kNT;        // hidden states per pass over the head
constexpr int kAhead = 8;                 // blocks of weights each lane has in flight
constexpr int kPadWords = 4;              // padding of a staged hidden state (spreads the banks)
constexpr int64_t kMaxD = 6144;           // staged hidden states must fit in shared memory

inline size_t smem_bytes(int64_t d) { return (size_t)kColsPass * (size_t)(d / 2 + kPadWords) * 4; }

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

// Logits of hidden states c0 .. c0 + kColsPass - 1 (fewer at the end) for
// every row of the packed head: logits[c][row] (bf16, round to nearest even
// from the fp32 sum).  Each warp takes whole tiles of 16 rows.
__global__ void __launch_bounds__(kThreads, 1)
    logits_kernel(const uint16_t *__restrict__ hidden, int64_t cols, int64_t d, const uint4 *__restrict__ wp,
                  const uint32_t *__restrict__ sp, int64_t rows, int64_t c0, uint16_t *__restrict__ logits)
{
    pdl_launch_dependents();
    pdl_wait();
    extern __shared__ uint32_t hs[];   // [kColsPass][d/2 + kPadWords]: bf16 pairs of each staged hidden state
    const int64_t words = d / 2, stride = words + kPadWords;
    const int nc = (int)(cols - c0 < kColsPass ? cols - c0 : kColsPass);
    for (int64_t i = threadIdx.x; i < kColsPass * words; i += kThreads) {
        const int c = (int)(i / words);
        const int64_t j = i - c * words;
        hs[c * stride + j] = c < nc ? __ldg(reinterpret_cast<const uint32_t *>(hidden + (c0 + c) * d) + j) : 0u;
    }
    __syncthreads();

    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5, g = lane >> 2, t = lane & 3;
    const int64_t tiles = rows / 16, nb = d / 64;
    const int64_t nwarps = (int64_t)gridDim.x * kWarps;
    const uint32_t kMask = 0x000F000Fu, kBias = 0x43004300u, kOff = 0x43084308u;   // 128 + n; 136 = 128 + 8
    const uint32_t *hrow[kNT];
#pragma unroll
    for (int n = 0; n < kNT; ++n) hrow[n] = hs + (n * 8 + g) * stride + t;

    for (int64_t T = (int64_t)blockIdx.x * kWarps + w; T < tiles; T += nwarps) {
        const uint4 *wt = wp + T * nb * 32 + lane;
        const uint32_t *st = sp + T * nb * 8 + g;
        float acc[kNT][4];
#pragma unroll
        for (int n = 0; n < kNT; ++n) acc[n][0] = acc[n][1] = acc[n][2] = acc[n][3] = 0.f;
        uint4 pw[kAhead];
        uint32_t ps[kAhead];
#pragma unroll
        for (int a = 0; a < kAhead; ++a) {
            pw[a] = a < nb ? __ldcs(wt + a * 32) : make_uint4(0, 0, 0, 0);
            ps[a] = a < nb ? __ldg(st + a * 8) : 0u;
        }
        for (int64_t B0 = 0; B0 < nb; B0 += kAhead) {
#pragma unroll
            for (int a = 0; a < kAhead; ++a) {
                const int64_t B = B0 + a;
                if (B < nb) {
                    const uint4 wv = pw[a];
                    const uint32_t sv = ps[a];
                    if (B + kAhead < nb) {   // refill this slot with the block kAhead ahead
                        pw[a] = __ldcs(wt + (B + kAhead) * 32);
                        ps[a] = __ldg(st + (B + kAhead) * 8);
                    }
                    float dd[kNT][4];
                    const uint32_t wds[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
                    for (int s = 0; s < 4; ++s) {
                        const uint32_t word = wds[s];
                        uint32_t ar[4];
#pragma unroll
                        for (int r = 0; r < 4; ++r) ar[r] = sub_bf16x2(lop3_and_or(word >> (4 * r), kMask, kBias), kOff);
                        const int64_t kw = (B * 64 + 16 * s) / 2;   // word offset of k in a staged row
#pragma unroll
                        for (int n = 0; n < kNT; ++n) mma_bf16(dd[n], ar, hrow[n][kw], hrow[n][kw + 4], s == 0);
                    }
                    const float s0 = f16_as_float(sv & 0xFFFFu), s1 = f16_as_float(sv >> 16);
#pragma unroll
                    for (int n = 0; n < kNT; ++n) {
                        acc[n][0] = fmaf(s0, dd[n][0], acc[n][0]);
                        acc[n][1] = fmaf(s0, dd[n][1], acc[n][1]);
                        acc[n][2] = fmaf(s1, dd[n][2], acc[n][2]);
                        acc[n][3] = fmaf(s1, dd[n][3], acc[n][3]);
                    }
                }
            }
        }
        const int64_t r0 = T * 16 + g, r1 = r0 + 8;
#pragma unroll
        for (int n = 0; n < kNT; ++n) {
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
