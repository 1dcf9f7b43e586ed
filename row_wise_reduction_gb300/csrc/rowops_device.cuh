// Device helpers shared by the rowops kernels: 16-byte streaming loads and
// stores, bf16 <-> fp32 conversion, fast exp2 / reciprocal, per-row geometry
// (unaligned head, 16-byte body, tail) and row-group reductions
// (__shfl_xor_sync butterflies plus a shared-memory combine across warps).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace rowops {

// ---------------------------------------------------------------------------
// element types: float, and bf16 carried as its 16-bit pattern
// ---------------------------------------------------------------------------
struct bf16_t {
    uint16_t bits;
};

template <typename T>
struct Elem;

template <>
struct Elem<float> {
    static constexpr int kBytes = 4;
    static constexpr int kVec = 4;  // elements per 16-byte vector
    __device__ __forceinline__ static float load(const float* p) { return *p; }
    __device__ __forceinline__ static void store(float* p, float v) { *p = v; }
    // 16-byte vector <-> fp32
    __device__ __forceinline__ static void unpack(const uint4& u, float* f) {
        f[0] = __uint_as_float(u.x);
        f[1] = __uint_as_float(u.y);
        f[2] = __uint_as_float(u.z);
        f[3] = __uint_as_float(u.w);
    }
    __device__ __forceinline__ static uint4 pack(const float* f) {
        return make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]), __float_as_uint(f[2]),
                          __float_as_uint(f[3]));
    }
    // v as this type stores it
    __device__ __forceinline__ static float round(float v) { return v; }
};

// two fp32 -> bf16x2, round to nearest even; `hi` lands in the upper half
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

template <>
struct Elem<bf16_t> {
    static constexpr int kBytes = 2;
    static constexpr int kVec = 8;
    __device__ __forceinline__ static float load(const bf16_t* p) {
        return __uint_as_float(uint32_t(p->bits) << 16);
    }
    __device__ __forceinline__ static void store(bf16_t* p, float v) {
        p->bits = uint16_t(pack_bf16x2(v, 0.f) & 0xffffu);
    }
    __device__ __forceinline__ static void unpack(const uint4& u, float* f) {
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            f[2 * i] = __uint_as_float(w[i] << 16);
            f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
        }
    }
    __device__ __forceinline__ static uint4 pack(const float* f) {
        return make_uint4(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]), pack_bf16x2(f[4], f[5]),
                          pack_bf16x2(f[6], f[7]));
    }
    __device__ __forceinline__ static float round(float v) { return __uint_as_float(pack_bf16x2(0.f, v) & 0xffff0000u); }
};

// ---------------------------------------------------------------------------
// 16-byte global accesses. Loads skip L1 allocation (every byte is read once)
// and ask L2 for 256-byte prefetch; stores are marked streaming (evict first).
// Plain coherent loads are used, not the read-only path, because x may equal y.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint4 ld_stream16(const void* p) {
    uint4 v;
    asm volatile("ld.global.L1::no_allocate.L2::256B.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ void st_stream16(void* p, const uint4& v) {
    asm volatile("st.global.cs.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z),
                 "r"(v.w)
                 : "memory");
}

// ---------------------------------------------------------------------------
// fast transcendental pieces (hardware approximations, flush-to-zero)
// ---------------------------------------------------------------------------
__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ float rcp_approx(float x) {
    float y;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

constexpr double kLog2e = 1.4426950408889634073599246810019;  // log2(e)
constexpr float kLog2eF = float(kLog2e);

// Packed fp32 pairs (sm_100 family): one instruction, two correctly rounded
// fp32 results, the same as two scalar add / mul / fma.
__device__ __forceinline__ float2 f2_add(float2 a, float2 b) {
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rd;\n\tmov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "add.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}
__device__ __forceinline__ float2 f2_mul(float2 a, float2 b) {
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rd;\n\tmov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "mul.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}
__device__ __forceinline__ float2 f2_fma(float2 a, float2 b, float2 c) {
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\tmov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "mov.b64 rc, {%6, %7};\n\tfma.rn.f32x2 rd, ra, rb, rc;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
    return d;
}
__device__ __forceinline__ float2 f2(float v) { return make_float2(v, v); }

// ---------------------------------------------------------------------------
// Row geometry: a row (or a segment of one) of n elements starting at byte
// address `addr` splits into `head` elements before the first 16-byte
// boundary, `nvec` whole 16-byte vectors and `tail` elements after them.
// Extra (head / tail) element e in [0, head + tail) has column
//   e < head ? e : head + nvec * kVec + (e - head).
// ---------------------------------------------------------------------------
struct RowGeom {
    int64_t nvec;
    int head;
    int tail;
    __device__ __forceinline__ int extras() const { return head + tail; }
};

template <typename T>
__device__ __forceinline__ RowGeom row_geometry(const void* row_ptr, int64_t n) {
    constexpr int B = Elem<T>::kBytes, V = Elem<T>::kVec;
    const unsigned mis = unsigned(reinterpret_cast<uintptr_t>(row_ptr) & 15u);
    int64_t head = mis ? int64_t((16u - mis) / B) : 0;
    if (head > n) head = n;
    RowGeom g;
    g.head = int(head);
    g.nvec = (n - head) / V;
    g.tail = int(n - head - g.nvec * V);
    return g;
}

__device__ __forceinline__ int64_t extra_col(const RowGeom& g, int e, int vec) {
    return e < g.head ? int64_t(e) : int64_t(g.head) + g.nvec * vec + (e - g.head);
}

// ---------------------------------------------------------------------------
// Row-group reductions. A row is owned by TPR consecutive threads of the CTA
// (TPR a power of two, 16..1024); the CTA holds BLOCK / TPR rows. Within a warp
// a butterfly of __shfl_xor_sync; for TPR > 32 each warp's value goes through
// shared memory (`red`, BLOCK / 32 floats) and every thread of the row combines
// the TPR / 32 values in the same fixed order. Every thread of the CTA must
// call these the same number of times (they contain __syncthreads when TPR > 32).
// Each call site must use its own `red` buffer: consecutive calls on the same
// buffer would need a second barrier.
// ---------------------------------------------------------------------------
struct OpMax {
    __device__ __forceinline__ float operator()(float a, float b) const { return fmaxf(a, b); }
};
struct OpSum {
    __device__ __forceinline__ float operator()(float a, float b) const { return a + b; }
};

template <int TPR, class Op>
__device__ __forceinline__ float group_reduce(float v, float* red, Op op) {
    constexpr int kLanes = TPR < 32 ? TPR : 32;
#pragma unroll
    for (int o = kLanes / 2; o > 0; o >>= 1) v = op(v, __shfl_xor_sync(0xffffffffu, v, o));
    if constexpr (TPR > 32) {
        constexpr int W = TPR / 32;
        const int warp = threadIdx.x >> 5;
        const int first = (warp / W) * W;  // first warp of this row
        if ((threadIdx.x & 31) == 0) red[warp] = v;
        __syncthreads();
        v = red[first];
#pragma unroll
        for (int i = 1; i < W; ++i) v = op(v, red[first + i]);
    }
    return v;
}

// Two sums reduced together (one butterfly, one barrier); `red` holds
// 2 * BLOCK / 32 floats.
template <int TPR>
__device__ __forceinline__ void group_reduce_sum2(float& a, float& b, float* red) {
    constexpr int kLanes = TPR < 32 ? TPR : 32;
#pragma unroll
    for (int o = kLanes / 2; o > 0; o >>= 1) {
        a += __shfl_xor_sync(0xffffffffu, a, o);
        b += __shfl_xor_sync(0xffffffffu, b, o);
    }
    if constexpr (TPR > 32) {
        constexpr int W = TPR / 32;
        const int warp = threadIdx.x >> 5;
        const int first = (warp / W) * W;
        if ((threadIdx.x & 31) == 0) {
            red[2 * warp] = a;
            red[2 * warp + 1] = b;
        }
        __syncthreads();
        a = red[2 * first];
        b = red[2 * first + 1];
#pragma unroll
        for (int i = 1; i < W; ++i) {
            a += red[2 * (first + i)];
            b += red[2 * (first + i) + 1];
        }
    }
}

// Online-softmax state (m, d): m the largest entry seen, d = sum exp(x - m).
// Merging two states [EX §2.5; L6 §7.2]: m = max(m1, m2),
//   d = d1 * exp(m1 - m) + d2 * exp(m2 - m); a state with d = 0 contributes nothing.
struct MD {
    float m, d;
};

__device__ __forceinline__ MD md_merge(MD a, MD b) {
    if (a.d == 0.f) return b;
    if (b.d == 0.f) return a;
    const float m = fmaxf(a.m, b.m);
    const float d = a.d * ex2_approx((a.m - m) * kLog2eF) + b.d * ex2_approx((b.m - m) * kLog2eF);
    return MD{m, d};
}

// Fold one value into a state.
__device__ __forceinline__ MD md_push(MD s, float x) {
    if (x == -INFINITY) return s;  // masked entry
    if (x > s.m) {
        s.d = s.d * ex2_approx((s.m - x) * kLog2eF) + 1.f;
        s.m = x;
    } else {
        s.d += ex2_approx((x - s.m) * kLog2eF);
    }
    return s;
}

// The same merge done as two cheap reductions: the group's max M with fmaxf,
// then sum_i d_i exp(m_i - M) (one exp per thread) -- instead of a tree of
// pairwise merges with two exps each. A NaN d_i stays NaN; states with d = 0
// contribute 0. Same fixed order on every call, so groups that merge the same
// values get the same (M, D). Uses the two buffers like two group_reduce calls.
template <int TPR>
__device__ __forceinline__ MD group_merge_fast(MD s, float* red_m, float* red_d) {
    const float M = group_reduce<TPR>(s.m, red_m, OpMax());
    const float d = s.d == 0.f ? 0.f : s.d * ex2_approx((s.m - M) * kLog2eF);
    return MD{M, group_reduce<TPR>(d, red_d, OpSum())};
}

template <int TPR>
__device__ __forceinline__ MD group_merge(MD s, float* red_m, float* red_d) {
    constexpr int kLanes = TPR < 32 ? TPR : 32;
#pragma unroll
    for (int o = kLanes / 2; o > 0; o >>= 1) {
        MD other{__shfl_xor_sync(0xffffffffu, s.m, o), __shfl_xor_sync(0xffffffffu, s.d, o)};
        s = md_merge(s, other);
    }
    if constexpr (TPR > 32) {
        constexpr int W = TPR / 32;
        const int warp = threadIdx.x >> 5;
        const int first = (warp / W) * W;
        if ((threadIdx.x & 31) == 0) {
            red_m[warp] = s.m;
            red_d[warp] = s.d;
        }
        __syncthreads();
        s = MD{red_m[first], red_d[first]};
#pragma unroll
        for (int i = 1; i < W; ++i) s = md_merge(s, MD{red_m[first + i], red_d[first + i]});
    }
    return s;
}

}  // namespace rowops
