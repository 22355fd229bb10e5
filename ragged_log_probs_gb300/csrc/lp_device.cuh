// Device helpers for the ragged log-probability kernels (sm_103a).
//
// Top-k ordering key, used at every merge level: fp32 logit descending, then token
// id ascending (ties on equal logits go to the lower id).  A warp keeps a sorted
// list of 32*SLOTS (logit, id) pairs, slot i = reg (i / 32), lane (i % 32).
#pragma once

#include <cstdint>
#include <utility>

namespace lpk {

constexpr unsigned kFull = 0xFFFFFFFFu;
constexpr float kLog2e = 1.4426950408889634f;
constexpr uint32_t kPadId = 0xFFFFFFFFu;

__device__ __forceinline__ float neg_inf() { return __int_as_float(0xff800000); }

// 2^x with the SFU (PTX ex2.approx; -inf -> +0).
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Streaming 16-byte load: read-only path, no L1 allocation, 256-byte L2 prefetch.
__device__ __forceinline__ float4 ldg_stream(const float* p) {
    float4 v;
    asm volatile("ld.global.nc.L1::no_allocate.L2::256B.v4.f32 {%0,%1,%2,%3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "l"(p));
    return v;
}

// Asynchronous 16-byte global -> shared copy (L1 bypass, 256-byte L2 prefetch) and
// its group bookkeeping. wait_group N returns once at most N of this thread's most
// recent groups are still in flight (a hardware wait, no polling loop).
__device__ __forceinline__ void cp_async16(uint32_t smem_addr, const float* gptr) {
    asm volatile("cp.async.cg.shared.global.L2::256B [%0], [%1], 16;" ::"r"(smem_addr), "l"(gptr) : "memory");
}
// U such copies of one lane: dst + 512*u <- src + 512*u bytes (a warp's 32 lanes fill
// 512 contiguous bytes per u), with the offsets as immediates of the instructions.
template <int OFF>
__device__ __forceinline__ void cp_async16_at(uint32_t dst, const float* src) {
    asm volatile("cp.async.cg.shared.global.L2::256B [%0+%2], [%1+%2], 16;" ::"r"(dst), "l"(src), "n"(OFF)
                 : "memory");
}
template <int... I>
__device__ __forceinline__ void cp_async16_seq(uint32_t dst, const float* src, std::integer_sequence<int, I...>) {
    (cp_async16_at<512 * I>(dst, src), ...);
}
template <int U>
__device__ __forceinline__ void cp_async16_run(uint32_t dst, const float* src) {
    cp_async16_seq(dst, src, std::make_integer_sequence<int, U>{});
}
// The same for a partial block: copies u with 32*u < n (n: the block's vectors left from
// this lane); the other slots get four -inf (a plain shared store, seen by this lane's
// later loads in program order).
__device__ __forceinline__ void sts_neg_inf4(uint32_t dst) {
    const uint32_t ni = 0xff800000u;
    asm volatile("st.shared.v4.b32 [%0], {%1, %1, %1, %1};" ::"r"(dst), "r"(ni) : "memory");
}
template <int... I>
__device__ __forceinline__ void cp_async16_seq_pad(uint32_t dst, const float* src, int n,
                                                   std::integer_sequence<int, I...>) {
    ((32 * I < n ? cp_async16_at<512 * I>(dst, src) : sts_neg_inf4(dst + 512 * I)), ...);
}
template <int U>
__device__ __forceinline__ void cp_async16_run_pad(uint32_t dst, const float* src, int n) {
    cp_async16_seq_pad(dst, src, n, std::make_integer_sequence<int, U>{});
}
// Asynchronous 4-byte global -> shared copy (an index or a status word fetched while
// the thread goes on; visible to it after its cp.async.wait_group).
__device__ __forceinline__ void cp_async4(uint32_t smem_addr, const void* gptr) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_addr), "l"(gptr) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Programmatic dependent launch: the producer lets the next kernel on the stream start
// launching; the consumer waits here until the producer has finished and its writes
// are visible (a no-op when the kernel was launched without the dependency).
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Bulk prefetch of the bytes [gptr, gptr + bytes) into L2, a hint with no completion to
// wait for (gptr 16-byte aligned, bytes a multiple of 16, the range inside one allocation).
__device__ __forceinline__ void prefetch_l2_bulk(const void* gptr, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(gptr), "r"(bytes) : "memory");
}

__device__ __forceinline__ bool better(float xa, uint32_t ia, float xb, uint32_t ib) {
    return xa > xb || (xa == xb && ia < ib);
}

// Order-preserving map float -> uint32 (atomicMax on a shared threshold word; 0 decodes
// to NaN, which fmaxf ignores, so a zeroed word means "no threshold yet").
__device__ __forceinline__ uint32_t f2ord(float f) {
    const uint32_t b = __float_as_uint(f);
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ float ord2f(uint32_t o) {
    return __uint_as_float((o & 0x80000000u) ? (o & 0x7FFFFFFFu) : ~o);
}

__device__ __forceinline__ float pick(const float4& v, int k) {
    return k == 0 ? v.x : (k == 1 ? v.y : (k == 2 ? v.z : v.w));
}

// Element mask of the vector whose first id is id0: the elements with id < end.
__device__ __forceinline__ uint32_t ids_below(uint32_t id0, uint32_t end) {
    const int n = (int)(end - id0);
    return n >= 4 ? 0xFu : (n <= 0 ? 0u : (1u << n) - 1u);
}

__device__ __forceinline__ uint32_t ge_mask(const float4& v, float thr) {
    return (uint32_t)(v.x >= thr) | ((uint32_t)(v.y >= thr) << 1) | ((uint32_t)(v.z >= thr) << 2) |
           ((uint32_t)(v.w >= thr) << 3);
}

// Descending bitonic merge of a bitonic 32-sequence held one element per lane.
__device__ __forceinline__ void bitonic_merge32(float& x, uint32_t& id, int lane) {
#pragma unroll
    for (int j = 16; j > 0; j >>= 1) {
        float ox = __shfl_xor_sync(kFull, x, j);
        uint32_t oid = __shfl_xor_sync(kFull, id, j);
        bool lower = (lane & j) == 0;
        bool ob = better(ox, oid, x, id);
        if (ob == lower) { x = ox; id = oid; }
    }
}

// Descending bitonic sort of 32 arbitrary pairs, one per lane.
__device__ __forceinline__ void bitonic_sort32(float& x, uint32_t& id, int lane) {
#pragma unroll
    for (int k = 2; k <= 32; k <<= 1) {
#pragma unroll
        for (int j = k >> 1; j > 0; j >>= 1) {
            float ox = __shfl_xor_sync(kFull, x, j);
            uint32_t oid = __shfl_xor_sync(kFull, id, j);
            bool lower = (lane & j) == 0;
            bool desc = (lane & k) == 0;
            bool ob = better(ox, oid, x, id);
            bool take = (lower == desc) ? ob : !ob;
            if (take) { x = ox; id = oid; }
        }
    }
}

// K-th largest (K <= 32) of one float per lane, broadcast to the warp: bitonic sort of
// the 32 values, descending, then lane K-1.
__device__ __forceinline__ float kth_largest32(float v, uint32_t K, int lane) {
#pragma unroll
    for (int k = 2; k <= 32; k <<= 1) {
#pragma unroll
        for (int j = k >> 1; j > 0; j >>= 1) {
            const float o = __shfl_xor_sync(kFull, v, j);
            const bool keep_max = ((lane & j) == 0) == ((lane & k) == 0);
            v = keep_max ? fmaxf(v, o) : fminf(v, o);
        }
    }
    return __shfl_sync(kFull, v, (K - 1) & 31);
}

// a := best 32*SLOTS of (a U b); both sorted descending in the lane-major layout.
template <int SLOTS>
__device__ __forceinline__ void merge_lists(float (&ax)[SLOTS], uint32_t (&ai)[SLOTS],
                                            const float (&bx)[SLOTS], const uint32_t (&bi)[SLOTS],
                                            int lane) {
    static_assert(SLOTS == 1 || SLOTS == 2, "one or two slots per lane");
    const int src = 31 - lane;
    if constexpr (SLOTS == 1) {
        float rx = __shfl_sync(kFull, bx[0], src);
        uint32_t ri = __shfl_sync(kFull, bi[0], src);
        if (better(rx, ri, ax[0], ai[0])) { ax[0] = rx; ai[0] = ri; }
        bitonic_merge32(ax[0], ai[0], lane);
    } else {
        // position i of the 64-list pairs with position 63-i of b:
        // slot lane <-> b slot 32+(31-lane); slot 32+lane <-> b slot (31-lane).
        float r1x = __shfl_sync(kFull, bx[1], src);
        uint32_t r1i = __shfl_sync(kFull, bi[1], src);
        float r0x = __shfl_sync(kFull, bx[0], src);
        uint32_t r0i = __shfl_sync(kFull, bi[0], src);
        float c0x = ax[0], c1x = ax[1];
        uint32_t c0i = ai[0], c1i = ai[1];
        if (better(r1x, r1i, c0x, c0i)) { c0x = r1x; c0i = r1i; }
        if (better(r0x, r0i, c1x, c1i)) { c1x = r0x; c1i = r0i; }
        // half-cleaner at distance 32 (same lane, two registers)
        if (better(c1x, c1i, c0x, c0i)) {
            float tx = c0x; c0x = c1x; c1x = tx;
            uint32_t ti = c0i; c0i = c1i; c1i = ti;
        }
        bitonic_merge32(c0x, c0i, lane);
        bitonic_merge32(c1x, c1i, lane);
        ax[0] = c0x; ai[0] = c0i;
        ax[1] = c1x; ai[1] = c1i;
    }
}

// a := best N of (a U b) for lists sorted descending in lanes 0..N-1 (N = 8, 16 or 32;
// the lanes of each other group of N work on their own entries, which nothing reads): the
// larger of a[l] and b[N-1-l] form a bitonic sequence holding the best N, which log2(N)
// half-cleaner stages sort.
template <int N>
__device__ __forceinline__ void merge_top(float& ax, uint32_t& ai, float bx, uint32_t bi, int lane) {
    static_assert(N == 8 || N == 16 || N == 32, "group of 8, 16 or 32 lanes");
    const int src = (lane & ~(N - 1)) | ((N - 1) - (lane & (N - 1)));
    const float rx = __shfl_sync(kFull, bx, src);
    const uint32_t ri = __shfl_sync(kFull, bi, src);
    if (better(rx, ri, ax, ai)) { ax = rx; ai = ri; }
#pragma unroll
    for (int j = N / 2; j > 0; j >>= 1) {
        const float ox = __shfl_xor_sync(kFull, ax, j);
        const uint32_t oid = __shfl_xor_sync(kFull, ai, j);
        const bool lower = (lane & j) == 0;
        if (better(ox, oid, ax, ai) == lower) { ax = ox; ai = oid; }
    }
}

// merge_top<N> with b already reversed: lane l holds b[(N-1) - (l mod N)] (loaded that
// way from shared memory, or sorted ascending), which saves merge_top's first shuffle.
template <int N>
__device__ __forceinline__ void merge_top_rev(float& ax, uint32_t& ai, float rx, uint32_t ri, int lane) {
    static_assert(N == 8 || N == 16 || N == 32, "group of 8, 16 or 32 lanes");
    if (better(rx, ri, ax, ai)) { ax = rx; ai = ri; }
#pragma unroll
    for (int j = N / 2; j > 0; j >>= 1) {
        const float ox = __shfl_xor_sync(kFull, ax, j);
        const uint32_t oid = __shfl_xor_sync(kFull, ai, j);
        const bool lower = (lane & j) == 0;
        if (better(ox, oid, ax, ai) == lower) { ax = ox; ai = oid; }
    }
}

// Packed fp32 pair arithmetic (one instruction for two lanes of data, sm_100+).
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\tmov.b64 rc, {%6, %7};\n\t"
        "fma.rn.ftz.f32x2 rd, ra, rb, rc;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
    return d;
}
__device__ __forceinline__ float2 fadd2(float2 a, float2 b) {
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "add.rn.ftz.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}

// max(a, b, c) in one instruction (three-source max, sm_100+).
__device__ __forceinline__ float max3(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

__device__ __forceinline__ float max4(const float4& v) { return fmaxf(max3(v.x, v.y, v.z), v.w); }

// Combine two (reference c, sum of 2^(x*log2e - c)) pairs in the log2 domain;
// c == -inf marks an empty sum.
__device__ __forceinline__ void lse2_combine(float& c, float& s, float oc, float os) {
    float C = fmaxf(c, oc);
    float a = (c == neg_inf()) ? 0.f : s * ex2(c - C);
    float b = (oc == neg_inf()) ? 0.f : os * ex2(oc - C);
    c = C;
    s = a + b;
}

__device__ __forceinline__ void warp_lse2_reduce(float& c, float& s) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        float oc = __shfl_xor_sync(kFull, c, o);
        float os = __shfl_xor_sync(kFull, s, o);
        lse2_combine(c, s, oc, os);
    }
}

}  // namespace lpk
