// Kernels of the ragged log-probability path.
//
//  k_plan   one CTA: output_row_offsets = [0, cumsum(echo ? len : 1)], validation,
//           clears the workspace status word and arrival counters.
//  k_rows   persistent stream-K reduction over all scored logits rows.
//
// The operation follows "MAX Python SDK 中 log_probabilities 模块解析" (sections
// "ragged 数据编排：从输入缓冲到 kernel 调用" and "top-k 语义：堆式 kernel 与「采样
// token 兜底」") and the logprob definition of "logprob、finish reason 与 output
// processing" (section "logprob 的数值形态").
#pragma once

#include <cstdint>

#include "lp_device.cuh"

namespace lpk {

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kPlanThreads = 1024;
constexpr uint32_t kStatusOffsets = 1u << 4;     // bit of LP_ERR_OFFSETS
constexpr uint32_t kStatusTokenRange = 1u << 5;  // bit of LP_ERR_TOKEN_RANGE

// Workspace: [header 256 B][counters u32 x g_max, padded to 256 B][partial slots].
struct WsHeader {
    uint32_t status;
    uint32_t rows;
    uint32_t reserved[62];
};

// Partial tuple of one piece of a split row (u32 words):
//   [0] max  [1] sum-exp  [2] target logit  [3] 1 if [2] is valid
//   [4, 4+K) top-k logits (sorted)   [4+K, 4+2K) their ids
__host__ __device__ inline uint32_t partial_stride_bytes(uint32_t K) {
    return ((4u + 2u * K) * 4u + 15u) & ~15u;
}

struct RowsParams {
    const float* logits;
    const uint32_t* off;
    const uint32_t* tokens;
    const uint32_t* sampled;
    const uint32_t* out_off;
    const uint8_t* echo;
    float* out_lp;
    uint32_t* out_tok;
    uint32_t* status;
    uint32_t* counters;
    unsigned char* partials;
    uint32_t T, V, B, K, W;
    uint32_t nq;          // 16-byte vectors per row in the stream-K space
    uint32_t stride;      // partial slot bytes
    uint32_t min_piece;   // minimum vectors per CTA
    uint32_t stage_offsets;  // 1: copy off/out_off to shared memory
};

// ---------------------------------------------------------------------------------
// Plan: one CTA, chunked block-wide exclusive scan.
__global__ void __launch_bounds__(kPlanThreads) k_plan(const uint32_t* __restrict__ off,
                                                       const uint8_t* __restrict__ echo, uint32_t B,
                                                       uint32_t T, uint32_t* __restrict__ out_off,
                                                       WsHeader* hdr, uint32_t* counters,
                                                       uint32_t n_counters) {
    __shared__ uint32_t s_warp[kPlanThreads / 32];
    __shared__ uint32_t s_carry;
    __shared__ uint32_t s_bad;
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    if (tid == 0) { s_carry = 0; s_bad = 0; }
    for (uint32_t i = tid; i < n_counters; i += kPlanThreads) counters[i] = 0;
    __syncthreads();
    for (uint32_t base = 0; base < B; base += kPlanThreads) {
        const uint32_t i = base + tid;
        uint32_t cnt = 0;
        bool bad = false;
        if (i < B) {
            uint32_t s = off[i], e = off[i + 1];
            if (e <= s || e > T) bad = true;
            else cnt = echo[i] ? (e - s) : 1u;
        }
        uint32_t x = cnt;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            uint32_t y = __shfl_up_sync(kFull, x, d);
            if (lane >= d) x += y;
        }
        if (lane == 31) s_warp[w] = x;
        if (bad) atomicOr(&s_bad, 1u);
        __syncthreads();
        if (w == 0) {
            uint32_t v = s_warp[lane];
#pragma unroll
            for (int d = 1; d < 32; d <<= 1) {
                uint32_t y = __shfl_up_sync(kFull, v, d);
                if (lane >= d) v += y;
            }
            s_warp[lane] = v;  // inclusive over warps
        }
        __syncthreads();
        const uint32_t incl = x + (w ? s_warp[w - 1] : 0u);
        if (i < B) out_off[i] = s_carry + incl - cnt;
        __syncthreads();
        if (tid == kPlanThreads - 1) s_carry += incl;
        __syncthreads();
    }
    if (tid == 0) {
        out_off[B] = s_carry;
        hdr->rows = s_carry;
        hdr->status = s_bad ? kStatusOffsets : 0u;
    }
}

// ---------------------------------------------------------------------------------
// Stream-K schedule over the vector space [0, R*nq): CTA c owns [start(c), start(c+1)).
__device__ __forceinline__ uint64_t sk_start(uint64_t c, uint64_t Q, uint64_t G) { return c * Q / G; }
// CTA that owns global vector g.
__device__ __forceinline__ uint64_t sk_owner(uint64_t g, uint64_t Q, uint64_t G) {
    return ((g + 1) * G - 1) / Q;
}

struct RowDesc {
    uint32_t r;      // logits row
    uint32_t t;      // target token
    bool valid;
};

template <int SLOTS, bool TOPK>
struct WarpTopK {
    float x[SLOTS];
    uint32_t id[SLOTS];
    __device__ __forceinline__ void reset() {
#pragma unroll
        for (int k = 0; k < SLOTS; ++k) { x[k] = neg_inf(); id[k] = kPadId; }
    }
};

template <int SLOTS, bool TOPK, int U>
struct alignas(16) RowsSmem {
    float cand_x[kWarps][64];
    uint32_t cand_i[kWarps][64];
    float list_x[kWarps][32 * SLOTS];
    uint32_t list_i[kWarps][32 * SLOTS];
    float red_m[kWarps];
    float red_s[kWarps];
    uint32_t thr;
    uint32_t last;
    float xt;
    uint32_t has_xt;
};

template <int SLOTS>
__device__ __forceinline__ float list_kth(const float (&x)[SLOTS], uint32_t K) {
    const uint32_t s = K - 1;
    float v = x[0];
    if constexpr (SLOTS == 2) v = (s >> 5) ? x[1] : x[0];
    return __shfl_sync(kFull, v, s & 31);
}

// Flush 32 buffered candidates of this warp into its sorted list.
template <int SLOTS>
__device__ __forceinline__ void flush32(float (&lx)[SLOTS], uint32_t (&li)[SLOTS], float* cx, uint32_t* ci,
                                        int cnt, int lane) {
    __syncwarp();
    float x = lane < cnt ? cx[lane] : neg_inf();
    uint32_t id = lane < cnt ? ci[lane] : kPadId;
    const bool more = lane + 32 < cnt;
    float mx = 0.f;
    uint32_t mi = 0;
    if (more) { mx = cx[lane + 32]; mi = ci[lane + 32]; }
    __syncwarp();
    if (more) { cx[lane] = mx; ci[lane] = mi; }
    __syncwarp();
    bitonic_sort32(x, id, lane);
    float bx[SLOTS];
    uint32_t bi[SLOTS];
    bx[0] = x; bi[0] = id;
    if constexpr (SLOTS == 2) { bx[1] = neg_inf(); bi[1] = kPadId; }
    merge_lists<SLOTS>(lx, li, bx, bi, lane);
}

// Load a stored partial's top-k into the lane-major list layout.
template <int SLOTS>
__device__ __forceinline__ void load_partial_list(const unsigned char* slot, uint32_t K, int lane,
                                                  float (&x)[SLOTS], uint32_t (&id)[SLOTS]) {
    const uint32_t* w = reinterpret_cast<const uint32_t*>(slot);
#pragma unroll
    for (int k = 0; k < SLOTS; ++k) {
        const uint32_t i = lane + 32 * k;
        if (i < K) {
            x[k] = __uint_as_float(__ldcg(w + 4 + i));
            id[k] = __ldcg(w + 4 + K + i);
        } else {
            x[k] = neg_inf();
            id[k] = kPadId;
        }
    }
}

template <int SLOTS, bool TOPK, int U>
__global__ void __launch_bounds__(kThreads) k_rows(RowsParams p) {
    extern __shared__ uint32_t s_dyn[];
    __shared__ RowsSmem<SLOTS, TOPK, U> sm;
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    const uint32_t B = p.B, V = p.V, K = p.K;

    if (__ldcg(p.status) & kStatusOffsets) return;  // plan rejected the offsets
    const uint32_t R = __ldcg(p.out_off + B);
    if (R == 0) return;
    if (R > p.T) {
        if (blockIdx.x == 0 && tid == 0) atomicOr(p.status, kStatusOffsets);
        return;
    }
    const uint64_t Q = (uint64_t)R * p.nq;
    uint64_t G = (Q + p.min_piece - 1) / p.min_piece;
    if (G > gridDim.x) G = gridDim.x;
    if (G == 0) G = 1;
    const uint64_t c = blockIdx.x;
    if (c >= G) return;

    const uint32_t* off = p.off;
    const uint32_t* out_off = p.out_off;
    if (p.stage_offsets) {
        for (uint32_t i = tid; i <= B; i += kThreads) {
            s_dyn[i] = p.off[i];
            s_dyn[B + 1 + i] = p.out_off[i];
        }
        __syncthreads();
        off = s_dyn;
        out_off = s_dyn + B + 1;
    }

    const uint64_t g0 = sk_start(c, Q, G), g1 = sk_start(c + 1, Q, G);
    uint32_t o = (uint32_t)(g0 / p.nq);
    const uint32_t o_first = o;
    uint32_t q0 = (uint32_t)(g0 - (uint64_t)o * p.nq);
    // batch of output row o: last b with out_off[b] <= o
    uint32_t lo = 0, hi = B;  // answer in [lo, hi)
    while (hi - lo > 1) {
        uint32_t mid = (lo + hi) >> 1;
        if (out_off[mid] <= o) lo = mid; else hi = mid;
    }
    uint32_t b = lo;

    float* cx = sm.cand_x[w];
    uint32_t* ci = sm.cand_i[w];

    for (uint64_t g = g0; g < g1;) {
        const uint32_t q1 = (uint32_t)min((uint64_t)p.nq, (uint64_t)q0 + (g1 - g));
        const bool full = (q0 == 0) && (q1 == p.nq);

        // ---- row descriptor -------------------------------------------------------
        RowDesc d;
        {
            const uint32_t ob = out_off[b], oe = out_off[b + 1];
            const uint32_t s = off[b], e = off[b + 1];
            const uint32_t cnt = oe - ob;
            const uint32_t len = e - s;
            const bool echo_b = p.echo[b] != 0;
            d.valid = (o >= ob) && (o < oe) && (e > s) && (e <= p.T) && (cnt == (echo_b ? len : 1u));
            d.r = 0;
            d.t = 0;
            if (d.valid) {
                d.r = e - cnt + (o - ob);
                d.t = (d.r + 1 < e) ? p.tokens[d.r + 1] : p.sampled[b];
            }
        }

        if (!d.valid) {
            if (q0 == 0 && tid < (int)p.W) {
                p.out_lp[(size_t)o * p.W + tid] = __int_as_float(0x7fc00000);
                p.out_tok[(size_t)o * p.W + tid] = kPadId;
            }
            if (q0 == 0 && tid == 0) atomicOr(p.status, kStatusOffsets);
        } else {
            const float* rowp = p.logits + (size_t)d.r * V;
            const int a = (int)(((uintptr_t)rowp >> 2) & 3u);
            const float* vbase = rowp - a;  // 16-byte aligned
            const uint32_t qf = a ? 1u : 0u;
            const uint32_t qe = (V + (uint32_t)a) >> 2;
            const uint32_t nfull = qe > qf ? qe - qf : 0u;

            // target logit: the piece whose elements cover t loads it
            const int64_t e_lo = 4 * (int64_t)q0 - a, e_hi = 4 * (int64_t)q1 - a;
            const bool t_here = d.t < V && (int64_t)d.t >= e_lo && (int64_t)d.t < e_hi;
            float xt = 0.f;
            if (t_here && tid == 0) xt = rowp[d.t];

            float m = neg_inf(), ms = 0.f, s = 0.f;
            float thr = neg_inf();
            int cnt = 0;
            WarpTopK<SLOTS, TOPK> L;
            L.reset();
            if (TOPK && tid == 0) sm.thr = f2ord(neg_inf());
            if (TOPK) __syncthreads();

            const uint32_t n = q1 - q0;
            for (uint32_t base = 0; base < n; base += kThreads * U) {
                float4 v[U];
                uint32_t vm[U];
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const uint32_t qi = base + u * kThreads + tid;
                    const uint32_t q = q0 + qi;
                    v[u] = make_float4(neg_inf(), neg_inf(), neg_inf(), neg_inf());
                    vm[u] = 0;
                    if (qi < n) {
                        if (q - qf < nfull) {
                            v[u] = ldg_stream(vbase + 4 * (size_t)q);
                            vm[u] = 0xFu;
                        } else {
                            float t4[4];
#pragma unroll
                            for (int k = 0; k < 4; ++k) {
                                const int64_t e = 4 * (int64_t)q - a + k;
                                t4[k] = neg_inf();
                                if (e >= 0 && e < (int64_t)V) { t4[k] = rowp[e]; vm[u] |= 1u << k; }
                            }
                            v[u] = make_float4(t4[0], t4[1], t4[2], t4[3]);
                        }
                    }
                }
                if (TOPK) thr = fmaxf(thr, ord2f(*(volatile uint32_t*)&sm.thr));
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const float4 x = v[u];
                    const float mx = fmaxf(fmaxf(x.x, x.y), fmaxf(x.z, x.w));
                    if (mx > m) {
                        s *= ex2((m - mx) * kLog2e);
                        m = mx;
                        ms = mx;
                    }
                    s += ex2((x.x - ms) * kLog2e) + ex2((x.y - ms) * kLog2e) +
                         ex2((x.z - ms) * kLog2e) + ex2((x.w - ms) * kLog2e);
                    if constexpr (TOPK) {
                        uint32_t pm = (mx >= thr) ? (ge_mask(x, thr) & vm[u]) : 0u;
                        unsigned any = __ballot_sync(kFull, pm != 0);
                        while (any) {
                            if (pm) {
                                const int k = __ffs(pm) - 1;
                                pm &= pm - 1;
                                const int slot = cnt + __popc(any & ((1u << lane) - 1u));
                                cx[slot] = pick(x, k);
                                ci[slot] = 4u * (q0 + base + u * kThreads + tid) - (uint32_t)a + (uint32_t)k;
                            }
                            cnt += __popc(any);
                            if (cnt >= 32) {
                                flush32<SLOTS>(L.x, L.id, cx, ci, cnt, lane);
                                cnt -= 32;
                                const float kth = list_kth<SLOTS>(L.x, K);
                                if (lane == 0) atomicMax(&sm.thr, f2ord(kth));
                                thr = fmaxf(thr, kth);
                                pm &= ge_mask(x, thr);
                            }
                            any = __ballot_sync(kFull, pm != 0);
                        }
                    }
                }
            }
            if constexpr (TOPK) {
                if (cnt > 0) flush32<SLOTS>(L.x, L.id, cx, ci, cnt, lane);
            }

            // ---- CTA combine: (m, s) and the warps' lists -> warp 0 ----------------
            warp_lse_reduce(m, s);
            if (lane == 0) { sm.red_m[w] = m; sm.red_s[w] = s; }
            if (tid == 0) { sm.xt = xt; sm.has_xt = t_here ? 1u : 0u; }
            if constexpr (TOPK) {
#pragma unroll
                for (int k = 0; k < SLOTS; ++k) {
                    sm.list_x[w][lane + 32 * k] = L.x[k];
                    sm.list_i[w][lane + 32 * k] = L.id[k];
                }
            }
            __syncthreads();
            if constexpr (TOPK) {
#pragma unroll
                for (int st = 1; st < kWarps; st <<= 1) {
                    if ((w & (2 * st - 1)) == 0) {
                        float bx[SLOTS];
                        uint32_t bi[SLOTS];
#pragma unroll
                        for (int k = 0; k < SLOTS; ++k) {
                            bx[k] = sm.list_x[w + st][lane + 32 * k];
                            bi[k] = sm.list_i[w + st][lane + 32 * k];
                        }
                        merge_lists<SLOTS>(L.x, L.id, bx, bi, lane);
#pragma unroll
                        for (int k = 0; k < SLOTS; ++k) {
                            sm.list_x[w][lane + 32 * k] = L.x[k];
                            sm.list_i[w][lane + 32 * k] = L.id[k];
                        }
                    }
                    __syncthreads();
                }
            }
            float M = neg_inf(), S = 0.f;
            if (w == 0) {
                M = lane < kWarps ? sm.red_m[lane] : neg_inf();
                S = lane < kWarps ? sm.red_s[lane] : 0.f;
                warp_lse_reduce(M, S);
            }

            bool emit = full;
            float xt_row = sm.xt;
            bool has_xt_row = sm.has_xt != 0;
            if (!full) {
                // ---- split row: publish this piece, the last arriving CTA merges -------
                const uint64_t gr = (uint64_t)o * p.nq;
                const uint64_t c0 = sk_owner(gr, Q, G), c1 = sk_owner(gr + p.nq - 1, Q, G);
                const uint32_t pieces = (uint32_t)(c1 - c0 + 1);
                unsigned char* my_slot = p.partials + (size_t)(2 * c + (o == o_first ? 0 : 1)) * p.stride;
                if (w == 0) {
                    uint32_t* pw = reinterpret_cast<uint32_t*>(my_slot);
                    if (lane == 0) {
                        pw[0] = __float_as_uint(M);
                        pw[1] = __float_as_uint(S);
                        pw[2] = __float_as_uint(xt_row);
                        pw[3] = has_xt_row ? 1u : 0u;
                    }
                    if constexpr (TOPK) {
#pragma unroll
                        for (int k = 0; k < SLOTS; ++k) {
                            const uint32_t i = lane + 32 * k;
                            if (i < K) { pw[4 + i] = __float_as_uint(L.x[k]); pw[4 + K + i] = L.id[k]; }
                        }
                    }
                    __threadfence();
                }
                __syncthreads();
                if (tid == 0) {
                    __threadfence();
                    const uint32_t ticket = atomicAdd(p.counters + c0, 1u);
                    sm.last = (ticket == pieces - 1) ? 1u : 0u;
                }
                __syncthreads();
                emit = sm.last != 0;
                if (emit) {
                    __threadfence();
                    // warp w folds pieces w, w + kWarps, ...
                    float pm_ = neg_inf(), ps_ = 0.f;
                    L.reset();
                    for (uint32_t j = w; j < pieces; j += kWarps) {
                        const uint64_t cc = c0 + j;
                        const uint32_t first_row = (uint32_t)(sk_start(cc, Q, G) / p.nq);
                        const unsigned char* slot = p.partials + (size_t)(2 * cc + (o == first_row ? 0 : 1)) * p.stride;
                        const uint32_t* pw = reinterpret_cast<const uint32_t*>(slot);
                        if (lane == 0) {
                            lse_combine(pm_, ps_, __uint_as_float(__ldcg(pw)), __uint_as_float(__ldcg(pw + 1)));
                            if (__ldcg(pw + 3)) { sm.xt = __uint_as_float(__ldcg(pw + 2)); sm.has_xt = 1u; }
                        }
                        if constexpr (TOPK) {
                            float bx[SLOTS];
                            uint32_t bi[SLOTS];
                            load_partial_list<SLOTS>(slot, K, lane, bx, bi);
                            merge_lists<SLOTS>(L.x, L.id, bx, bi, lane);
                        }
                    }
                    if (lane == 0) { sm.red_m[w] = pm_; sm.red_s[w] = ps_; }
                    if constexpr (TOPK) {
#pragma unroll
                        for (int k = 0; k < SLOTS; ++k) {
                            sm.list_x[w][lane + 32 * k] = L.x[k];
                            sm.list_i[w][lane + 32 * k] = L.id[k];
                        }
                    }
                    __syncthreads();
                    if constexpr (TOPK) {
#pragma unroll
                        for (int st = 1; st < kWarps; st <<= 1) {
                            if ((w & (2 * st - 1)) == 0) {
                                float bx[SLOTS];
                                uint32_t bi[SLOTS];
#pragma unroll
                                for (int k = 0; k < SLOTS; ++k) {
                                    bx[k] = sm.list_x[w + st][lane + 32 * k];
                                    bi[k] = sm.list_i[w + st][lane + 32 * k];
                                }
                                merge_lists<SLOTS>(L.x, L.id, bx, bi, lane);
#pragma unroll
                                for (int k = 0; k < SLOTS; ++k) {
                                    sm.list_x[w][lane + 32 * k] = L.x[k];
                                    sm.list_i[w][lane + 32 * k] = L.id[k];
                                }
                            }
                            __syncthreads();
                        }
                    }
                    if (w == 0) {
                        M = lane < kWarps ? sm.red_m[lane] : neg_inf();
                        S = lane < kWarps ? sm.red_s[lane] : 0.f;
                        warp_lse_reduce(M, S);
                    }
                    xt_row = sm.xt;
                    has_xt_row = sm.has_xt != 0;
                    if (tid == 0) p.counters[c0] = 0u;  // ready for the next call
                }
            }

            // ---- write the row: K top columns + the target column -----------------
            if (emit && w == 0) {
                const double lse = (double)M + (double)logf(S);
                const size_t ro = (size_t)o * p.W;
                if constexpr (TOPK) {
#pragma unroll
                    for (int k = 0; k < SLOTS; ++k) {
                        const uint32_t i = lane + 32 * k;
                        if (i < K) {
                            p.out_lp[ro + i] = (float)((double)L.x[k] - lse);
                            p.out_tok[ro + i] = L.id[k];
                        }
                    }
                }
                if (lane == 0) {
                    float lpt = __int_as_float(0x7fc00000);
                    if (d.t < V && has_xt_row) lpt = (float)((double)xt_row - lse);
                    if (d.t >= V) atomicOr(p.status, kStatusTokenRange);
                    p.out_lp[ro + K] = lpt;
                    p.out_tok[ro + K] = d.t;
                }
            }
        }
        __syncthreads();

        // ---- next piece -------------------------------------------------------------
        g += q1 - q0;
        q0 = 0;
        ++o;
        while (b + 1 < B && out_off[b + 1] <= o) ++b;
    }
}

}  // namespace lpk
