// FP8 prep kernel: r = x D H_d / sqrt(d) (Q and K, mode 1), then per block
// of 128 tokens of one (batch, head): amax, scale = amax / 448, e4m3 codes
// of r / scale.  FlashAttention-3 deep-reading report §2.2 and §3.3 (block
// quantization; incoherent processing with M = diag(+-1) x Hadamard, O(d log d)).
//
// One CTA owns one 128-token block of one head, so the block amax is a CTA
// reduction and the data is read once and written once (the op is bound by
// device-memory bandwidth).  A warp holds whole rows: lane l keeps elements
// [l*E, l*E + E) of a row, E = d / 32.  The Walsh-Hadamard butterflies with
// stride < E stay inside a thread; the wider ones pair lanes with shuffles.
// With RoPE (rotary position embedding; Su et al., "RoFormer", 2021) the
// row is first turned pair by pair with the caller's binary32 cos / sin
// tables (N, d/2): a' = a cos - b sin, b' = a sin + b cos, each product and
// sum rounded (no FMA), pairs (i, i + d/2) ("half-split": the partner sits
// 16 lanes away) or (2i, 2i + 1) ("interleaved": inside the thread).  This is
// the placement the report's §2.2 names: quantisation riding inside the
// memory-bound rotary-embedding pass.
// Mode 2 (one scale per tensor) runs three launches: block amax into
// `scales`, a one-CTA reduction that turns them into the tensor's scale,
// and the quantisation with that scale.
#include <cuda_bf16.h>

#include <cstdint>

#include "fp8_prep.cuh"
#include "sm103_ptx.cuh"

namespace attn {
namespace {

constexpr int kBlockRows = 128;

// Sign c of the +-1 diagonal: bit 63 of splitmix64 output c for state
// `seed` (output c is the mixing function applied to seed + (c + 1) * gamma).
__device__ __forceinline__ float diag_sign(unsigned long long seed, int c) {
    unsigned long long z = seed + static_cast<unsigned long long>(c + 1) * 0x9E3779B97F4A7C15ull;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    z ^= z >> 31;
    return (z >> 63) ? -1.0f : 1.0f;
}

enum Pass { kFused = 0, kAmaxOnly = 1, kApplyScale = 2 };
enum Rope { kNoRope = 0, kRopeHalf = 1, kRopeInterleaved = 2 };

template <int K> struct FloatVec;
template <> struct FloatVec<1> { using T = float; };
template <> struct FloatVec<2> { using T = float2; };
template <> struct FloatVec<4> { using T = float4; };
template <> struct FloatVec<8> { using T = float4; };   // loaded as two float4

// K consecutive floats from a 4*K-byte aligned address.
template <int K>
__device__ __forceinline__ void load_floats(const float* __restrict__ p, float (&out)[K]) {
    if constexpr (K == 8) {
        const float4 a = __ldg(reinterpret_cast<const float4*>(p));
        const float4 b = __ldg(reinterpret_cast<const float4*>(p) + 1);
        out[0] = a.x; out[1] = a.y; out[2] = a.z; out[3] = a.w;
        out[4] = b.x; out[5] = b.y; out[6] = b.z; out[7] = b.w;
    } else {
        const typename FloatVec<K>::T v = __ldg(reinterpret_cast<const typename FloatVec<K>::T*>(p));
        const float* f = reinterpret_cast<const float*>(&v);
#pragma unroll
        for (int k = 0; k < K; ++k) out[k] = f[k];
    }
}

// x / s rounded to nearest for s > 0, from the correctly rounded reciprocal
// and one residual correction (Markstein, "Computation of elementary
// functions on the IBM RISC System/6000 processor", IBM J. R&D 1990): with
// inv = RN(1/s), q0 = RN(x * inv) and the exact residual x - q0 * s (one FMA),
// q0 + residual * inv rounds to RN(x / s) for the normal-range quotients
// here (|x / s| <= 448).  The sign is copied so that -0 / s stays -0.
__device__ __forceinline__ float div_by_scale(float x, float s, float inv) {
    const float q0 = x * inv;
    const float rem = fmaf(-q0, s, x);
    return copysignf(fmaf(rem, inv, q0), x);
}

template <int E> struct RowLoad;
template <> struct RowLoad<2> { using T = uint32_t; };
template <> struct RowLoad<4> { using T = uint2; };
template <> struct RowLoad<8> { using T = uint4; };

template <int D, int WARPS, int PASS, int ROPE>
__global__ void __launch_bounds__(WARPS * 32)
    fp8_prep_kernel(const __nv_bfloat16* __restrict__ x, uint8_t* __restrict__ x8, float* __restrict__ scales,
                    int H, int N, int nblk, int rotate, unsigned long long seed,
                    const float* __restrict__ rope_cos, const float* __restrict__ rope_sin) {
    constexpr int E = D / 32;                     // elements per lane
    // table entries a lane needs per row: E (half-split) or E/2 (interleaved)
    constexpr int TE = ROPE == kRopeInterleaved ? E / 2 : E;
    constexpr int RPW = kBlockRows / WARPS;       // rows per warp
    using Raw = typename RowLoad<E>::T;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int blk = blockIdx.x % nblk;
    const int bh = blockIdx.x / nblk;
    const int b = bh / H, h = bh % H;
    const int n0 = blk * kBlockRows + warp * RPW;

    // Issue every row load of this thread before any arithmetic.
    Raw raw[RPW];
#pragma unroll
    for (int rr = 0; rr < RPW; ++rr) {
        const int n = n0 + rr;
        if (n < N) {
            raw[rr] = __ldg(reinterpret_cast<const Raw*>(x + ((static_cast<size_t>(b) * N + n) * H + h) * D + lane * E));
        } else {
            raw[rr] = Raw{};
        }
    }

    // RoPE table entries of this lane's pairs: loaded up front for all rows
    // where the registers allow it (d <= 128), else row by row.
    constexpr bool PRELOAD = ROPE != kNoRope && D <= 128;
    constexpr int TROWS = PRELOAD ? RPW : 1;
    const int i0 = ROPE == kRopeHalf ? (lane & 15) * E : lane * (E / 2);   // first pair index
    float tc[TROWS][TE], ts[TROWS][TE];
    auto load_table = [&](int rr, int slot) {
        const int n = min(n0 + rr, N - 1);
        load_floats<TE>(rope_cos + static_cast<size_t>(n) * (D / 2) + i0, tc[slot]);
        load_floats<TE>(rope_sin + static_cast<size_t>(n) * (D / 2) + i0, ts[slot]);
    };
    if constexpr (PRELOAD) {
#pragma unroll
        for (int rr = 0; rr < RPW; ++rr) load_table(rr, rr);
    }

    float sgn[E];
#pragma unroll
    for (int e = 0; e < E; ++e) sgn[e] = rotate ? diag_sign(seed, lane * E + e) : 1.0f;

    float r[RPW][E];
    float amax = 0.0f;
#pragma unroll
    for (int rr = 0; rr < RPW; ++rr) {
        const __nv_bfloat162* pv = reinterpret_cast<const __nv_bfloat162*>(&raw[rr]);
#pragma unroll
        for (int k = 0; k < E / 2; ++k) {
            r[rr][2 * k] = __bfloat162float(pv[k].x);
            r[rr][2 * k + 1] = __bfloat162float(pv[k].y);
        }
        const int slot = PRELOAD ? rr : 0;
        if constexpr (ROPE != kNoRope && !PRELOAD) load_table(rr, 0);
        if constexpr (ROPE == kRopeHalf) {
            // lanes 0-15 hold the first halves a, lanes 16-31 the partners b
            const bool upper = lane >= 16;
#pragma unroll
            for (int e = 0; e < E; ++e) {
                const float other = __shfl_xor_sync(0xffffffffu, r[rr][e], 16);
                const float a = upper ? other : r[rr][e], bb = upper ? r[rr][e] : other;
                const float c = tc[slot][e], sn = ts[slot][e];
                r[rr][e] = upper ? __fadd_rn(__fmul_rn(a, sn), __fmul_rn(bb, c))
                                 : __fsub_rn(__fmul_rn(a, c), __fmul_rn(bb, sn));
            }
        } else if constexpr (ROPE == kRopeInterleaved) {
#pragma unroll
            for (int k = 0; k < E / 2; ++k) {
                const float a = r[rr][2 * k], bb = r[rr][2 * k + 1];
                const float c = tc[slot][k], sn = ts[slot][k];
                r[rr][2 * k] = __fsub_rn(__fmul_rn(a, c), __fmul_rn(bb, sn));
                r[rr][2 * k + 1] = __fadd_rn(__fmul_rn(a, sn), __fmul_rn(bb, c));
            }
        }
        if (rotate) {
#pragma unroll
            for (int e = 0; e < E; ++e) r[rr][e] *= sgn[e];
            // Butterflies inside the thread (strides 1 .. E/2).
#pragma unroll
            for (int st = 1; st < E; st <<= 1) {
#pragma unroll
                for (int e = 0; e < E; ++e) {
                    if ((e & st) == 0) {
                        const float a = r[rr][e], c = r[rr][e + st];
                        r[rr][e] = a + c;
                        r[rr][e + st] = a - c;
                    }
                }
            }
            // Butterflies across lanes (strides E .. D/2).
#pragma unroll
            for (int ls = 1; ls < 32; ls <<= 1) {
                const bool upper = (lane & ls) != 0;
#pragma unroll
                for (int e = 0; e < E; ++e) {
                    const float other = __shfl_xor_sync(0xffffffffu, r[rr][e], ls);
                    r[rr][e] = upper ? (other - r[rr][e]) : (r[rr][e] + other);
                }
            }
            constexpr float inv_sqrt_d = D == 64 ? 0.125f : (D == 128 ? 0.08838834764831845f : 0.0625f);
            // "+ 0.0f" maps a -0 produced by a sign flip of an exact zero to +0,
            // so a zero always encodes as the +0 code.
#pragma unroll
            for (int e = 0; e < E; ++e) r[rr][e] = __fadd_rn(r[rr][e] * inv_sqrt_d, 0.0f);
        }
#pragma unroll
        for (int e = 0; e < E; ++e) amax = fmaxf(amax, fabsf(r[rr][e]));
    }

    __shared__ float warp_max[WARPS];
    __shared__ float block_scale;
    if constexpr (PASS != kApplyScale) {
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
        if (lane == 0) warp_max[warp] = amax;
        __syncthreads();
        if (threadIdx.x == 0) {
            float a = warp_max[0];
#pragma unroll
            for (int w = 1; w < WARPS; ++w) a = fmaxf(a, warp_max[w]);
            if constexpr (PASS == kAmaxOnly) {
                scales[static_cast<size_t>(bh) * nblk + blk] = a;
            } else {
                const float sc = a > 0.0f ? __fdiv_rn(a, 448.0f) : 1.0f;
                scales[static_cast<size_t>(bh) * nblk + blk] = sc;
                block_scale = sc;
            }
        }
        if constexpr (PASS == kAmaxOnly) return;
        __syncthreads();
    } else {
        if (threadIdx.x == 0) block_scale = scales[static_cast<size_t>(bh) * nblk + blk];
        __syncthreads();
    }
    const float sc = block_scale;
    const float inv = __frcp_rn(sc);
#pragma unroll
    for (int rr = 0; rr < RPW; ++rr) {
        const int n = n0 + rr;
        if (n >= N) continue;
        uint8_t* dst = x8 + ((static_cast<size_t>(b) * N + n) * H + h) * D + lane * E;
        float y[E];
#pragma unroll
        for (int e = 0; e < E; ++e) y[e] = div_by_scale(r[rr][e], sc, inv);
        if constexpr (E == 2) {
            uint16_t v;
            asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(v) : "f"(y[1]), "f"(y[0]));
            *reinterpret_cast<uint16_t*>(dst) = v;
        } else if constexpr (E == 4) {
            *reinterpret_cast<uint32_t*>(dst) = pack_e4m3x4(y[0], y[1], y[2], y[3]);
        } else {
            uint2 v;
            v.x = pack_e4m3x4(y[0], y[1], y[2], y[3]);
            v.y = pack_e4m3x4(y[4], y[5], y[6], y[7]);
            *reinterpret_cast<uint2*>(dst) = v;
        }
    }
}

// Mode 2: the block maxima in `scales` -> one scale, written to every entry.
__global__ void __launch_bounds__(1024) per_tensor_scale_kernel(float* scales, long long count) {
    float a = 0.0f;
    for (long long i = threadIdx.x; i < count; i += blockDim.x) a = fmaxf(a, scales[i]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, off));
    __shared__ float wm[32];
    __shared__ float result;
    if ((threadIdx.x & 31) == 0) wm[threadIdx.x >> 5] = a;
    __syncthreads();
    if (threadIdx.x == 0) {
        float m = 0.0f;
        for (int w = 0; w < static_cast<int>(blockDim.x >> 5); ++w) m = fmaxf(m, wm[w]);
        result = m > 0.0f ? __fdiv_rn(m, 448.0f) : 1.0f;
    }
    __syncthreads();
    const float s = result;
    for (long long i = threadIdx.x; i < count; i += blockDim.x) scales[i] = s;
}

template <int D, int WARPS, int ROPE>
cudaError_t launch_prep(const void* x, void* x8, float* scales, int B, int H, int N, int mode,
                        unsigned long long seed, bool is_v, const float* rope_cos, const float* rope_sin,
                        cudaStream_t stream) {
    const int nblk = (N + kBlockRows - 1) / kBlockRows;
    const long long ctas = static_cast<long long>(B) * H * nblk;
    if (ctas >= (1ll << 31)) return cudaErrorInvalidValue;
    const auto* xb = static_cast<const __nv_bfloat16*>(x);
    auto* q8 = static_cast<uint8_t*>(x8);
    const int rotate = (mode == 1 && !is_v) ? 1 : 0;
    const dim3 grid(static_cast<unsigned>(ctas)), block(WARPS * 32);
    if (mode != 2) {
        fp8_prep_kernel<D, WARPS, kFused, ROPE>
            <<<grid, block, 0, stream>>>(xb, q8, scales, H, N, nblk, rotate, seed, rope_cos, rope_sin);
        return cudaGetLastError();
    }
    fp8_prep_kernel<D, WARPS, kAmaxOnly, ROPE>
        <<<grid, block, 0, stream>>>(xb, q8, scales, H, N, nblk, 0, seed, rope_cos, rope_sin);
    per_tensor_scale_kernel<<<1, 1024, 0, stream>>>(scales, ctas);
    fp8_prep_kernel<D, WARPS, kApplyScale, ROPE>
        <<<grid, block, 0, stream>>>(xb, q8, scales, H, N, nblk, 0, seed, rope_cos, rope_sin);
    return cudaGetLastError();
}

template <int D, int WARPS>
cudaError_t launch_prep_any(const void* x, void* x8, float* scales, int B, int H, int N, int mode,
                            unsigned long long seed, bool is_v, const float* rope_cos, const float* rope_sin,
                            int rope, cudaStream_t stream) {
    switch (rope) {
        case kNoRope:
            return launch_prep<D, WARPS, kNoRope>(x, x8, scales, B, H, N, mode, seed, is_v, nullptr, nullptr, stream);
        case kRopeHalf:
            return launch_prep<D, WARPS, kRopeHalf>(x, x8, scales, B, H, N, mode, seed, is_v, rope_cos, rope_sin,
                                                    stream);
        case kRopeInterleaved:
            return launch_prep<D, WARPS, kRopeInterleaved>(x, x8, scales, B, H, N, mode, seed, is_v, rope_cos,
                                                           rope_sin, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

cudaError_t run_fp8_prep(const void* x, void* x8, float* scales, int B, int H, int N, int d, int mode,
                         unsigned long long sign_seed, bool is_v, const float* rope_cos, const float* rope_sin,
                         int rope, cudaStream_t stream) {
    switch (d) {
        case 64:
            return launch_prep_any<64, 16>(x, x8, scales, B, H, N, mode, sign_seed, is_v, rope_cos, rope_sin, rope,
                                           stream);
        case 128:
            return launch_prep_any<128, 16>(x, x8, scales, B, H, N, mode, sign_seed, is_v, rope_cos, rope_sin, rope,
                                            stream);
        case 256:
            return launch_prep_any<256, 32>(x, x8, scales, B, H, N, mode, sign_seed, is_v, rope_cos, rope_sin, rope,
                                            stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace attn
