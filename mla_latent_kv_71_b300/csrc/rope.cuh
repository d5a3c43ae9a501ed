// rope.cuh -- the rotary position embedding of the decoupled RoPE part of
// the key and the query ([Mishra] "Step 4: decoupled RoPE"; [llms] "The
// Positional Problem and Decoupled RoPE"), shared by the prologue's
// finishing kernels and the GEMM epilogue that writes the query directly.
//
// RoPE rotates pair (x_2k, x_2k+1) of a d_r-vector by pos * base^(-2k/d_r)
// (the pages fix only that the angle grows with the position; pairing and
// frequencies are the common reading).  The angle is kept in turns: the host
// passes each frequency f_k = base^(-2k/d_r) / 2pi as a 64-bit fixed-point
// fraction F_k = round(f_k 2^64), and pos * F_k taken modulo 2^64 is the
// fraction of a turn pos * f_k mod 1, exact up to pos times the rounding of
// F_k (below 2^-33 of a turn for any int32 position).  Its top 24 bits,
// rounded, give the angle to 2^-25 of a turn (2e-7 rad), and sin / cos come
// from fp32 sincospif, whose argument needs no further reduction.  So
// positions in the hundreds of thousands keep their phase without fp64
// arithmetic (slow on this GPU).
#pragma once

#include <cstdint>

namespace mla {
namespace rope {

constexpr int MAX_PAIRS = 64;  // d_r <= 128

// sin and cos of the angle pos * f, f given as the 0.64 fixed-point
// fraction of a turn described above.
__device__ __forceinline__ void rope_sincos(int64_t pos, uint64_t f, float& sn, float& cs) {
    const uint64_t t = static_cast<uint64_t>(pos) * f;  // fraction of a turn, mod 1
    const uint32_t top = static_cast<uint32_t>((t + (1ull << 39)) >> 40);  // 24 bits, rounded
    sincospif(2.0f * (static_cast<float>(top) * 0x1p-24f), &sn, &cs);
}

// (a, b) rotated by the angle whose sine and cosine are sn, cs.
__device__ __forceinline__ void rotate(float a, float b, float sn, float cs, float& ya, float& yb) {
    ya = fmaf(a, cs, -b * sn);
    yb = fmaf(a, sn, b * cs);
}

}  // namespace rope
}  // namespace mla
