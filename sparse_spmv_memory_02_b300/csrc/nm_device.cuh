// Device helpers shared by the libnm kernels: streaming loads, byte
// permutes, mixed-precision FMA and warp reductions (sm_103a).
#pragma once

#include <cuda_fp16.h>
#include <stdint.h>

namespace nm {

// ---------------------------------------------------------------- loads
// Weights are streamed once per call: bypass L1 and ask L2 for 256-byte
// lines so that consecutive 16-byte requests of a warp share DRAM bursts.
__device__ __forceinline__ uint4 ld_stream_v4(const uint4 *p)
{
    uint4 r;
    asm("ld.global.nc.L1::no_allocate.L2::256B.v4.u32 {%0, %1, %2, %3}, [%4];"
        : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
        : "l"(p));
    return r;
}

__device__ __forceinline__ uint32_t ld_stream_u8(const uint8_t *p)
{
    uint16_t r;
    asm("ld.global.nc.L1::no_allocate.u8 %0, [%1];" : "=h"(r) : "l"(p));
    return r;
}

__device__ __forceinline__ uint32_t ld_stream_u16(const uint16_t *p)
{
    uint16_t r;
    asm("ld.global.nc.L1::no_allocate.u16 %0, [%1];" : "=h"(r) : "l"(p));
    return r;
}

__device__ __forceinline__ uint32_t ld_stream_u32(const uint32_t *p)
{
    uint32_t r;
    asm("ld.global.nc.L1::no_allocate.u32 %0, [%1];" : "=r"(r) : "l"(p));
    return r;
}

__device__ __forceinline__ uint64_t ld_stream_u64(const uint64_t *p)
{
    uint64_t r;
    asm("ld.global.nc.L1::no_allocate.u64 %0, [%1];" : "=l"(r) : "l"(p));
    return r;
}

// Activations are small and reused by every warp of the SM: keep them in L1.
__device__ __forceinline__ uint4 ld_keep_v4(const uint4 *p)
{
    uint4 r;
    asm("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];"
        : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
        : "l"(p));
    return r;
}

// ---------------------------------------------------------------- bits
// Byte permute: result byte i = byte (sel >> 4i) & 7 of the 8-byte {hi, lo}.
// Every selector in this library keeps bit 3 of each nibble clear, so the
// PTX instruction is used as is: __byte_perm ignores that bit by definition,
// which costs a masking instruction per permute whose selector is not a
// compile-time constant.  Bits 16-31 of sel are ignored.
// The bit helpers below also compile for the host (the same results, so the
// mask decode can be checked on a machine without a GPU).
__host__ __device__ __forceinline__ uint32_t prmt(uint32_t lo, uint32_t hi, uint32_t sel)
{
#ifdef __CUDA_ARCH__
    uint32_t r;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(lo), "r"(hi), "r"(sel));
    return r;
#else
    const uint64_t b = (static_cast<uint64_t>(hi) << 32) | lo;
    uint32_t r = 0;
    for (int i = 0; i < 4; ++i)
        r |= static_cast<uint32_t>((b >> (8 * ((sel >> (4 * i)) & 7u))) & 0xFFu) << (8 * i);
    return r;
#endif
}

#ifdef __CUDA_ARCH__
__device__ __forceinline__ uint32_t ctz(uint32_t v) { return __ffs(v) - 1; }   // v != 0
__device__ __forceinline__ uint32_t msb(uint32_t v) { return 31 - __clz(v); }  // v != 0
#else
inline uint32_t ctz(uint32_t v) { return static_cast<uint32_t>(__builtin_ctz(v)); }
inline uint32_t msb(uint32_t v) { return 31u - static_cast<uint32_t>(__builtin_clz(v)); }
#endif

// Selector that gathers fp16 lanes pa and pb (0..3) of the 8-byte pair
// {hi, lo} into the low and high half of a 32-bit word.
__host__ __device__ __forceinline__ uint32_t sel_pair(uint32_t pa, uint32_t pb)
{
    return 0x1010u + 0x22u * pa + 0x2200u * pb;
}

// fp16 lanes pa and pb (0..7) of the four words {d, c, b, a} -> one half2.
// Two permutes take the lanes' positions within each half of the group, a
// third picks the half each lane lives in.
__host__ __device__ __forceinline__ uint32_t gather_pair8(uint32_t a, uint32_t b, uint32_t c,
                                                          uint32_t d, uint32_t pa, uint32_t pb)
{
    const uint32_t s = sel_pair(pa & 3u, pb & 3u);
    const uint32_t lo = prmt(a, b, s);
    const uint32_t hi = prmt(c, d, s);
    const uint32_t pick = ((pa & 4u) ? 0x54u : 0x10u) | ((pb & 4u) ? 0x7600u : 0x3200u);
    return prmt(lo, hi, pick);
}

// ---------------------------------------------------------------- math
// acc + v.lo*x.lo + v.hi*x.hi with fp16 operands and fp32 accumulation.
// The product of two fp16 values is exact in fp32, so each step rounds once
// (on the host too, where fmaf of the converted operands does the same).
__host__ __device__ __forceinline__ float fma_h2(uint32_t v, uint32_t x, float acc)
{
#if defined(__CUDA_ARCH__) && NM_USE_MIXED_FMA
    asm("{\n\t.reg .f16 vl, vh, xl, xh;\n\t"
        "mov.b32 {vl, vh}, %1;\n\t"
        "mov.b32 {xl, xh}, %2;\n\t"
        "fma.rn.f32.f16 %0, vl, xl, %0;\n\t"
        "fma.rn.f32.f16 %0, vh, xh, %0;\n\t}"
        : "+f"(acc)
        : "r"(v), "r"(x));
    return acc;
#else
    // the halves by value (no pointer cast: the host compiler's aliasing
    // rules forbid reading a uint32_t through a __half2)
    const float vl = __half2float(__ushort_as_half(static_cast<unsigned short>(v & 0xFFFFu)));
    const float vh = __half2float(__ushort_as_half(static_cast<unsigned short>(v >> 16)));
    const float xl = __half2float(__ushort_as_half(static_cast<unsigned short>(x & 0xFFFFu)));
    const float xh = __half2float(__ushort_as_half(static_cast<unsigned short>(x >> 16)));
    acc = fmaf(vl, xl, acc);
    return fmaf(vh, xh, acc);
#endif
}

// ---------------------------------------------------------------- reduce
// Reduce V (a power of two <= 32) per-lane partial sums across the warp so
// that afterwards v[0] of lane l holds the warp total of index
// (l >> (5 - log2 V)).  Each halving stage exchanges half of the live values,
// so V sums cost V-1 shuffles instead of 5 V.  Stage n (live values) and o
// (shuffle distance) are template arguments so every index is constant.
template <int n, int o, int V>
__device__ __forceinline__ void reduce_scatter_stage(float (&v)[V], int lane)
{
    if constexpr (o >= 1) {
        if constexpr (n > 1) {
            const bool upper = (lane & o) != 0;
#pragma unroll
            for (int i = 0; i < n / 2; ++i) {
                const float send = upper ? v[i] : v[i + n / 2];
                const float keep = upper ? v[i + n / 2] : v[i];
                v[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
            }
            reduce_scatter_stage<n / 2, o / 2, V>(v, lane);
        } else {
            v[0] += __shfl_xor_sync(0xffffffffu, v[0], o);
            reduce_scatter_stage<1, o / 2, V>(v, lane);
        }
    }
}

template <int V>
__device__ __forceinline__ void warp_reduce_scatter(float (&v)[V], int lane)
{
    static_assert(V >= 1 && V <= 32 && (V & (V - 1)) == 0, "V must be a power of two <= 32");
    reduce_scatter_stage<V, 16, V>(v, lane);
}

template <int V>
__host__ __device__ constexpr int log2i() { return V <= 1 ? 0 : 1 + log2i<V / 2>(); }

__host__ __device__ constexpr int pow2_ceil(int v)
{
    return v <= 1 ? 1 : 2 * pow2_ceil((v + 1) / 2);
}

__device__ __forceinline__ void store_y(void *y, int64_t idx, float v, bool f32)
{
    if (f32)
        static_cast<float *>(y)[idx] = v;
    else
        static_cast<__half *>(y)[idx] = __float2half_rn(v);
}

}  // namespace nm
