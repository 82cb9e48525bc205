// Logits-form cross entropy: memory-bound row kernels for sm_103a.
//
// Forward (Transformer Engine parallel_cross_entropy, API card "Description":
// fused online softmax + cross entropy, FP32 loss for BF16/FP32 logits; pull
// request #3273 "Changes": the single-GPU path is one forward kernel that
// saves per-row statistics instead of the derivative):
//   one CTA per row streams the row once with 16-byte vector loads, keeps a
//   running (max, sum of exp) per thread, merges them with warp shuffles and a
//   shared-memory pass, and writes the row loss and (max, lse).
// Backward (same pull request: the gradient is rebuilt from the saved stats):
//   one CTA per row streams the logits once more and writes
//   dz = g (exp(z - lse) - (1 - eps) onehot(y) - eps / V), zeros for ignored rows.
// Mean reduction: one CTA sums the per-row losses in a fixed order (run to run
// identical) and counts the rows whose target is not ignore_idx.
// Fused forward + backward (for a caller that knows grad_output up front): each
// row is read from HBM once and its gradient written once; the second read of
// the row is served by L2.  Rows up to 16 KiB: several CTAs per SM, each asking
// L2 for its next row ahead of time.  Longer rows: one to four persistent CTAs
// per SM whose producer thread streams the rows through a shared-memory ring
// with TMA bulk copies.

#include "vce_internal.cuh"
#include "sm100_ptx.cuh"

#include <math.h>
#include <mutex>

namespace vce {
namespace {

// ---------------------------------------------------------------------------
// element access
// ---------------------------------------------------------------------------

template <typename T> struct Elem;
template <> struct Elem<float> {
    static constexpr int kVec = 4;  // elements per 16-byte vector
    __device__ static float load1(const float* p) { return __ldcs(p); }
    __device__ static void unpack(const uint4& u, float (&v)[4]) {
        v[0] = __uint_as_float(u.x); v[1] = __uint_as_float(u.y);
        v[2] = __uint_as_float(u.z); v[3] = __uint_as_float(u.w);
    }
    __device__ static uint4 pack(const float (&v)[4]) {
        return make_uint4(__float_as_uint(v[0]), __float_as_uint(v[1]),
                          __float_as_uint(v[2]), __float_as_uint(v[3]));
    }
    __device__ static void store1(float* p, float x) { *p = x; }
    // largest of the U vectors' elements: a tree of fmaxf (kTree: shorter
    // dependency chain) or a chain (fewer live registers); a maximum is exact, so
    // both give the same value
    template <int U, bool kTree>
    __device__ static float max_raw(const uint4 (&raw)[U]) {
        float f[4 * U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            f[4 * u] = __uint_as_float(raw[u].x); f[4 * u + 1] = __uint_as_float(raw[u].y);
            f[4 * u + 2] = __uint_as_float(raw[u].z); f[4 * u + 3] = __uint_as_float(raw[u].w);
        }
        if constexpr (kTree) {
#pragma unroll
            for (int n = 2 * U; n >= 1; n >>= 1)
#pragma unroll
                for (int i = 0; i < n; ++i) f[i] = fmaxf(f[i], f[i + n]);
        } else {
#pragma unroll
            for (int i = 1; i < 4 * U; ++i) f[0] = fmaxf(f[0], f[i]);
        }
        return f[0];
    }
};
template <> struct Elem<__nv_bfloat16> {
    static constexpr int kVec = 8;
    __device__ static float load1(const __nv_bfloat16* p) {
        unsigned short b = __ldcs(reinterpret_cast<const unsigned short*>(p));
        return __uint_as_float(uint32_t(b) << 16);
    }
    __device__ static void unpack(const uint4& u, float (&v)[8]) {
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            v[2 * i] = __uint_as_float(w[i] << 16);
            v[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
        }
    }
    __device__ static uint32_t pack2(float lo, float hi) {
        __nv_bfloat162 b = __floats2bfloat162_rn(lo, hi);
        return *reinterpret_cast<uint32_t*>(&b);
    }
    __device__ static uint4 pack(const float (&v)[8]) {
        return make_uint4(pack2(v[0], v[1]), pack2(v[2], v[3]), pack2(v[4], v[5]), pack2(v[6], v[7]));
    }
    __device__ static void store1(__nv_bfloat16* p, float x) { *p = __float2bfloat16_rn(x); }
    // largest of the U vectors' elements: max.bf16x2 on the packed words, as a
    // tree (kTree: shorter dependency chain) or a chain (fewer live registers),
    // then the larger of the last word's two halves.  A BF16 maximum is exact, so
    // this is the FP32 maximum of the unpacked values either way.
    template <int U, bool kTree>
    __device__ static float max_raw(const uint4 (&raw)[U]) {
        uint32_t w[4 * U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            w[4 * u] = raw[u].x; w[4 * u + 1] = raw[u].y; w[4 * u + 2] = raw[u].z; w[4 * u + 3] = raw[u].w;
        }
        if constexpr (kTree) {
#pragma unroll
            for (int n = 2 * U; n >= 1; n >>= 1)
#pragma unroll
                for (int i = 0; i < n; ++i) asm("max.bf16x2 %0, %1, %2;" : "=r"(w[i]) : "r"(w[i]), "r"(w[i + n]));
        } else {
#pragma unroll
            for (int i = 1; i < 4 * U; ++i) asm("max.bf16x2 %0, %1, %2;" : "=r"(w[0]) : "r"(w[0]), "r"(w[i]));
        }
        return fmaxf(__uint_as_float(w[0] << 16), __uint_as_float(w[0] & 0xFFFF0000u));
    }
};

// v[k] = g * exp2(v[k] * log2(e) + negl) - b for a vector of K (even) elements,
// two lanes per FFMA2: each lane is the same IEEE fused multiply-add as fmaf.
template <int K>
__device__ __forceinline__ void grad_lanes(float (&v)[K], float g, float negl, float b) {
    static_assert(K % 2 == 0, "pairs of lanes");
    const float2 l2 = make_float2(kLog2e, kLog2e), nl = make_float2(negl, negl);
    const float2 g2 = make_float2(g, g), nb = make_float2(-b, -b);
#pragma unroll
    for (int k = 0; k < K; k += 2) {
        const float2 a = __ffma2_rn(make_float2(v[k], v[k + 1]), l2, nl);
        const float2 d = __ffma2_rn(g2, make_float2(ex2f(a.x), ex2f(a.y)), nb);
        v[k] = d.x;
        v[k + 1] = d.y;
    }
}

// Split of a row into a scalar head (up to the first 16-byte boundary), whole
// 16-byte vectors and a scalar tail.
template <typename T>
struct RowSplit {
    int64_t head, nvec, tail0;
    __device__ RowSplit(const T* p, int64_t vocab) {
        const uintptr_t a = reinterpret_cast<uintptr_t>(p);
        head = int64_t((16 - (a & 15)) & 15) / int64_t(sizeof(T));
        if (head > vocab) head = vocab;
        nvec = (vocab - head) / Elem<T>::kVec;
        tail0 = head + nvec * Elem<T>::kVec;
    }
};

// Checks of the bounds-checking build (VCE_BOUNDS; constant true otherwise):
// element j of a row lies in [0, vocab); vector i of the row's 16-byte interior
// lies inside the row and its address ``a`` is 16-byte aligned.
__device__ __forceinline__ bool elem_ok(int64_t j, int64_t vocab, int* st) {
    return VCE_BOUNDS(j >= 0 && j < vocab, st);
}
template <typename T>
__device__ __forceinline__ bool vec_ok(const RowSplit<T>& sp, int64_t i, int64_t vocab, const void* a, int* st) {
    return VCE_BOUNDS(i >= 0 && i < sp.nvec && sp.head + (i + 1) * Elem<T>::kVec <= vocab && aligned16(a), st);
}

// Writes a row of zeros (the gradient of an ignored row or of a bad target).
template <int THREADS, typename T>
__device__ __forceinline__ void row_zero(T* q, const RowSplit<T>& sp, int64_t vocab, int* st) {
    using E = Elem<T>;
    if (threadIdx.x < sp.head && elem_ok(threadIdx.x, vocab, st)) E::store1(q + threadIdx.x, 0.f);
    uint4* qv = reinterpret_cast<uint4*>(q + sp.head);
    for (int64_t i = threadIdx.x; i < sp.nvec; i += THREADS)
        if (vec_ok(sp, i, vocab, qv + i, st)) qv[i] = make_uint4(0, 0, 0, 0);
    for (int64_t j = sp.tail0 + threadIdx.x; j < vocab; j += THREADS)
        if (elem_ok(j, vocab, st)) E::store1(q + j, 0.f);
}

// Writes zeros over one CTA's share of a row: 16-byte vectors [v0, v1) of the
// row's interior, with the head elements before it (``head``) and the tail
// elements after it (``tail``).
template <int NT, typename T>
__device__ __forceinline__ void part_zero(T* q, const RowSplit<T>& sp, int64_t vocab, int64_t v0, int64_t v1,
                                          bool head, bool tail, int* st) {
    using E = Elem<T>;
    if (head && threadIdx.x < sp.head && elem_ok(threadIdx.x, vocab, st)) E::store1(q + threadIdx.x, 0.f);
    uint4* qv = reinterpret_cast<uint4*>(q + sp.head);
    for (int64_t i = v0 + threadIdx.x; i < v1; i += NT)
        if (vec_ok(sp, i, vocab, qv + i, st)) qv[i] = make_uint4(0, 0, 0, 0);
    if (tail)
        for (int64_t j = sp.tail0 + threadIdx.x; j < vocab; j += NT)
            if (elem_ok(j, vocab, st)) E::store1(q + j, 0.f);
}

// ---------------------------------------------------------------------------
// online softmax accumulator: s = sum exp(z - m) over the values seen
// ---------------------------------------------------------------------------

struct OnlineLse {
    float m = -INFINITY;   // running max
    float negm = 0.f;      // -m * log2(e), 0 while m = -inf
    float s = 0.f;         // sum of exp(z - m)
    float sum = 0.f;       // sum of z (label smoothing term)

    // raises the running max to vm if that is larger, rescaling s
    __device__ __forceinline__ void raise(float vm) {
        if (vm > m) {
            s = s * ex2f((m - vm) * kLog2e);  // s = 0 while m = -inf: stays 0
            m = vm;
            negm = -vm * kLog2e;
        }
    }

    template <int K, bool kSum>
    __device__ __forceinline__ void push(const float (&v)[K]) {
        float vm = v[0];
#pragma unroll
        for (int i = 1; i < K; ++i) vm = fmaxf(vm, v[i]);
        raise(vm);
        add<K, kSum>(v);
    }

    // adds the K values to s (and sum); none of them exceeds m
    template <int K, bool kSum>
    __device__ __forceinline__ void add(const float (&v)[K]) {
        if constexpr (K % 2 == 0) {
            // two lanes per instruction (FFMA2 / FADD2): exponent arguments and the
            // running sums of even and odd elements
            const float2 l2 = make_float2(kLog2e, kLog2e), nm = make_float2(negm, negm);
            float2 t2 = make_float2(0.f, 0.f);
#pragma unroll
            for (int i = 0; i < K; i += 2) {
                const float2 a = __ffma2_rn(make_float2(v[i], v[i + 1]), l2, nm);
                t2 = __fadd2_rn(t2, make_float2(ex2f(a.x), ex2f(a.y)));
            }
            s += t2.x + t2.y;
            if (kSum) {
                float2 u2 = make_float2(0.f, 0.f);
#pragma unroll
                for (int i = 0; i < K; i += 2) u2 = __fadd2_rn(u2, make_float2(v[i], v[i + 1]));
                sum += u2.x + u2.y;
            }
        } else {
            float t = 0.f;
#pragma unroll
            for (int i = 0; i < K; ++i) t += ex2f(fmaf(v[i], kLog2e, negm));
            s += t;
            if (kSum) {
                float u = 0.f;
#pragma unroll
                for (int i = 0; i < K; ++i) u += v[i];
                sum += u;
            }
        }
    }

    // merge another (m2, s2) pair into this one
    __device__ __forceinline__ void merge(float m2, float s2, float sum2) {
        const float mn = fmaxf(m, m2);
        sum += sum2;
        if (mn == -INFINITY) { m = mn; s = 0.f; return; }
        s = s * ex2f((m - mn) * kLog2e) + s2 * ex2f((m2 - mn) * kLog2e);
        m = mn;
    }
};

// Folds U whole vectors into the accumulator, kGroup at a time: one max over a
// group's elements (from the packed values), one rescale, then every element's
// exponent with the same offset, so a group's arithmetic has no branch inside
// and interleaves.  The short-row fused kernel and the 128-thread forward fold
// their vectors in pairs this way (2-3% faster on rows of 4096-8000 BF16
// elements), with the same grouping, so their results stay equal bit for bit.
// The other kernels fold one vector at a time with OnlineLse::push: pairs
// measured 1% slower at V = 128256 and 2% faster or slower between 24000 and
// 100352 depending on the length.
template <typename T, int U, bool kSum, bool kTree, int kGroup>
__device__ __forceinline__ void push_raw(OnlineLse& acc, const uint4 (&raw)[U]) {
    using E = Elem<T>;
    static_assert(U % kGroup == 0, "whole groups");
#pragma unroll
    for (int g = 0; g < U; g += kGroup) {
        const uint4(&grp)[kGroup] = *reinterpret_cast<const uint4(*)[kGroup]>(&raw[g]);
        acc.raise(E::template max_raw<kGroup, kTree>(grp));
#pragma unroll
        for (int u = 0; u < kGroup; ++u) {
            float v[E::kVec];
            E::unpack(grp[u], v);
            acc.template add<E::kVec, kSum>(v);
        }
    }
}

// Warp-wide max of an FP32 value in one instruction (redux.sync, sm_100 family).
__device__ __forceinline__ float warp_max(float x) {
    float r;
    asm("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(r) : "f"(x));
    return r;
}

// Combines the 32 lanes' (m, s, sum) of a warp, max first: the warp's max M in
// one step, each lane's s rescaled to it once (s e^(m - M), 0 for a lane that
// saw nothing), then the rescaled sums added over a butterfly, so no exponent
// waits on a shuffle.  Every lane ends with the same result.
template <bool kSum>
__device__ __forceinline__ void warp_combine(OnlineLse& a) {
    const float mx = warp_max(a.m);
    float s = a.m == -INFINITY ? 0.f : a.s * ex2f((a.m - mx) * kLog2e);
    float u = a.sum;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        s += __shfl_xor_sync(0xffffffffu, s, off);
        if (kSum) u += __shfl_xor_sync(0xffffffffu, u, off);
    }
    a.m = mx;
    a.s = s;
    a.sum = u;
}

// Combines the partials of a CTA's W warps: each warp combines its lanes, lane
// 0 of each writes the warp's partial to shared memory, and warp 0 combines
// those; ``sync`` is the barrier of the participating threads.  Thread 0 holds
// the result.
template <int W, bool kSum, typename Sync>
__device__ __forceinline__ void group_merge(OnlineLse& a, float* sm_m, float* sm_s, float* sm_sum, Sync sync) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    warp_combine<kSum>(a);
    if (lane == 0) { sm_m[warp] = a.m; sm_s[warp] = a.s; sm_sum[warp] = a.sum; }
    sync();
    if (warp == 0) {
        OnlineLse b;
        if (lane < W) { b.m = sm_m[lane]; b.s = sm_s[lane]; b.sum = sm_sum[lane]; }
        warp_combine<kSum>(b);
        a = b;
    }
}

// As group_merge, but every warp ends with the combined result, so no second
// barrier is needed to share it.  ``sm`` holds two sets of W partials (6 x 32
// floats) and ``set`` (0 or 1) picks the one this merge uses: callers alternate
// it from one merge to the next, so a warp that runs ahead into the next merge
// writes the other set while slower warps still read this one, and it cannot
// reach the merge after that before every warp has passed the next merge's
// barrier.  Each warp combines all W partials with warp 0's operations of
// group_merge in the same order, so every thread holds the same bits as thread
// 0 of group_merge over the same partials.
template <int W, bool kSum, typename Sync>
__device__ __forceinline__ void group_merge_all(OnlineLse& a, float* sm, uint32_t set, Sync sync) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    float* pm = sm + set * 96;
    warp_combine<kSum>(a);
    if (lane == 0) { pm[warp] = a.m; pm[32 + warp] = a.s; pm[64 + warp] = a.sum; }
    sync();
    OnlineLse b;
    if (lane < W) { b.m = pm[lane]; b.s = pm[32 + lane]; b.sum = pm[64 + lane]; }
    warp_combine<kSum>(b);
    a = b;
}

template <int THREADS, bool kSum>
__device__ __forceinline__ void block_merge(OnlineLse& a, float* sm_m, float* sm_s, float* sm_sum) {
    group_merge<THREADS / 32, kSum>(a, sm_m, sm_s, sm_sum, [] { __syncthreads(); });
}

// ---------------------------------------------------------------------------
// K1: forward row kernel
// ---------------------------------------------------------------------------

template <int THREADS, int MINB, typename T, bool kSmooth>
__global__ void __launch_bounds__(THREADS, MINB)
ce_forward_rows(const T* __restrict__ logits, int64_t n_rows, int64_t vocab, int64_t stride,
                const int64_t* __restrict__ target, float eps, int64_t ignore_idx,
                float* __restrict__ loss_rows, float2* __restrict__ stats, int* dev_status) {
    using E = Elem<T>;
    constexpr int V = E::kVec;
    constexpr int U = 4;  // vectors in flight per thread per iteration
    __shared__ float sm_m[32], sm_s[32], sm_sum[32];

    for (int64_t row = blockIdx.x; row < n_rows; row += gridDim.x) {
        const int64_t y = target[row];
        if (y == ignore_idx) {
            if (threadIdx.x == 0) {
                loss_rows[row] = 0.f;
                stats[row] = make_float2(0.f, 0.f);
            }
            continue;
        }
        const T* p = logits + row * stride;
        const RowSplit<T> sp(p, vocab);
        // With 512 threads the target logit is requested now and used after the
        // merge, so its latency overlaps the row's stream (0.4% faster at BF16 V =
        // 50257 and 128256).  The extra live registers cost more than that in the
        // 128- and 256-thread kernels (1.5% slower at V = 4096, 3% at 32000), which
        // load it after the merge.
        const bool y_in = y >= 0 && y < vocab;
        constexpr bool kEarlyY = THREADS >= 512;
        const float zy_early = (kEarlyY && threadIdx.x == 0 && y_in) ? E::load1(p + y) : 0.f;
        OnlineLse acc;
        if (threadIdx.x < sp.head && elem_ok(threadIdx.x, vocab, dev_status)) {
            float v[1] = {E::load1(p + threadIdx.x)};
            acc.push<1, kSmooth>(v);
        }
        const uint4* pv = reinterpret_cast<const uint4*>(p + sp.head);
        int64_t i = threadIdx.x;
        for (; i + (U - 1) * THREADS < sp.nvec; i += U * THREADS) {
            uint4 raw[U];
#pragma unroll
            for (int u = 0; u < U; ++u)
                raw[u] = vec_ok(sp, i + u * THREADS, vocab, pv + i + u * THREADS, dev_status)
                             ? __ldcs(pv + i + u * THREADS) : make_uint4(0, 0, 0, 0);
            if constexpr (THREADS == 128) {
                push_raw<T, U, kSmooth, false, 2>(acc, raw);  // a chain: 32 registers
            } else {
                // one vector at a time, as the ring kernels fold them
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    float v[V];
                    E::unpack(raw[u], v);
                    acc.push<V, kSmooth>(v);
                }
            }
        }
        for (; i < sp.nvec; i += THREADS) {
            float v[V];
            E::unpack(vec_ok(sp, i, vocab, pv + i, dev_status) ? __ldcs(pv + i) : make_uint4(0, 0, 0, 0), v);
            acc.push<V, kSmooth>(v);
        }
        for (int64_t j = sp.tail0 + threadIdx.x; j < vocab; j += THREADS) {
            float v[1] = {elem_ok(j, vocab, dev_status) ? E::load1(p + j) : 0.f};
            acc.push<1, kSmooth>(v);
        }
        block_merge<THREADS, kSmooth>(acc, sm_m, sm_s, sm_sum);
        if (threadIdx.x == 0) {
            const float lse = acc.m + logf(acc.s);
            float loss;
            if (y_in) {
                const float zy = kEarlyY ? zy_early : E::load1(p + y);
                loss = lse - zy;
                if (kSmooth) loss = (1.f - eps) * loss + eps * (lse - acc.sum / float(vocab));
            } else {
                loss = __int_as_float(0x7fc00000);  // NaN
                report(dev_status, VCE_DEVSTATUS_BAD_TARGET);
            }
            loss_rows[row] = loss;
            stats[row] = make_float2(acc.m, lse);
        }
        __syncthreads();  // shared scratch reused by the next row
    }
}

// ---------------------------------------------------------------------------
// K2: backward row kernel (dlogits may alias logits)
// ---------------------------------------------------------------------------

template <int THREADS, typename T>
__global__ void __launch_bounds__(THREADS)
ce_backward_rows(const T* logits, int64_t n_rows, int64_t vocab, int64_t stride,
                 const int64_t* __restrict__ target, const float2* __restrict__ stats,
                 const int64_t* __restrict__ n_valid, const float* __restrict__ grad_output,
                 float eps, int reduce_loss, int64_t ignore_idx, T* dlogits, int* dev_status) {
    using E = Elem<T>;
    constexpr int V = E::kVec;
    constexpr int U = 2;

    for (int64_t row = blockIdx.x; row < n_rows; row += gridDim.x) {
        const int64_t y = target[row];
        T* q = dlogits + row * stride;
        const T* p = logits + row * stride;
        const RowSplit<T> sp(q, vocab);
        const bool ignored = (y == ignore_idx);
        const bool bad = !ignored && (y < 0 || y >= vocab);
        if (ignored || bad) {
            if (bad && threadIdx.x == 0) report(dev_status, VCE_DEVSTATUS_BAD_TARGET);
            row_zero<THREADS, T>(q, sp, vocab, dev_status);
            continue;
        }
        const float g = upstream_grad(reduce_loss, grad_output, n_valid, row);
        const Exp2Offset eo = exp2_offset(stats[row].y);
        const float negl = eo.neg;
        const float gp = g * eo.fix;              // scale of the softmax term
        const float b = g * eps / float(vocab);   // eps / V share of every class
        const float c = g * (1.f - eps);          // target class

        auto grad1 = [&](int64_t j) {
            if (!elem_ok(j, vocab, dev_status)) return;
            const float z = E::load1(p + j);
            float d = fmaf(gp, ex2f(fmaf(z, kLog2e, negl)), -b);
            if (j == y) d = __fsub_rn(d, c);  // never contracted with c's product: the vector path's value
            E::store1(q + j, d);
        };
        if (threadIdx.x < sp.head) grad1(threadIdx.x);
        const uint4* pv = reinterpret_cast<const uint4*>(p + sp.head);
        uint4* qv = reinterpret_cast<uint4*>(q + sp.head);
        auto gradv = [&](const uint4& raw, int64_t i) {
            float v[V];
            E::unpack(raw, v);
            grad_lanes<V>(v, gp, negl, b);
            const int64_t base = sp.head + i * V;
            if (uint64_t(y - base) < uint64_t(V)) {
#pragma unroll
                for (int k = 0; k < V; ++k) v[k] = __fsub_rn(v[k], (base + k == y) ? c : 0.f);
            }
            if (vec_ok(sp, i, vocab, qv + i, dev_status)) __stcs(qv + i, E::pack(v));
        };
        int64_t i = threadIdx.x;
        for (; i + (U - 1) * THREADS < sp.nvec; i += U * THREADS) {
            uint4 raw[U];
#pragma unroll
            for (int u = 0; u < U; ++u)
                raw[u] = vec_ok(sp, i + u * THREADS, vocab, pv + i + u * THREADS, dev_status)
                             ? __ldcs(pv + i + u * THREADS) : make_uint4(0, 0, 0, 0);
#pragma unroll
            for (int u = 0; u < U; ++u) gradv(raw[u], i + u * THREADS);
        }
        for (; i < sp.nvec; i += THREADS)
            gradv(vec_ok(sp, i, vocab, pv + i, dev_status) ? __ldcs(pv + i) : make_uint4(0, 0, 0, 0), i);
        for (int64_t j = sp.tail0 + threadIdx.x; j < vocab; j += THREADS) grad1(j);
    }
}

// ---------------------------------------------------------------------------
// K8: mean over non-ignored rows (fixed summation order)
// ---------------------------------------------------------------------------

constexpr int kMeanThreads = 1024;

// Adds the compensated pair (h2, l2) to (hi, lo) with TwoSum, so the pair keeps
// the rounding error of every addition; an infinite or NaN sum propagates alone.
__device__ __forceinline__ void pair_add(float& hi, float& lo, float h2, float l2) {
    const float s = hi + h2;
    if (!isfinite(s)) {
        hi = s;
        lo = 0.f;
        return;
    }
    const float bb = s - hi;
    const float e = (hi - (s - bb)) + (h2 - bb);
    const float l = lo + l2 + e;
    hi = s + l;
    lo = l - (hi - s);
}

// kCounted: N_v was counted before (the fused call's count), read from
// ``n_valid``; only the losses are loaded.
template <bool kCounted>
__global__ void __launch_bounds__(kMeanThreads)
mean_loss_kernel(const float* __restrict__ loss_rows, const int64_t* __restrict__ target,
                 int64_t n, int64_t ignore_idx, int reduce, float* __restrict__ loss_out,
                 int64_t* __restrict__ n_valid) {
    __shared__ float sm_h[32], sm_l[32];
    __shared__ long long sm_c[32];
    // Each thread adds its rows eight at a time (a small FP32 tree per batch of
    // loads) into a running FP32 sum with Neumaier compensation (the rounding
    // error each addition dropped is kept and added back), which keeps it within
    // FP32 rounding of the exact total.  The 1024 per-thread (sum, error) pairs
    // are then combined in a fixed order by TwoSum additions, which carry the
    // error along as FP64 additions would, in FP32 arithmetic: FP64 runs at a
    // small fraction of the FP32 rate on this GPU (an FP64 combine took 8.2 us
    // per launch at 16384 rows against 6.1 us, and converting and adding every
    // row in FP64 took 14 us for 16384 rows and 585 us for 1M rows).
    float fs = 0.f, fc = 0.f;
    int ci = 0;  // this thread's count (at most n / 1024 + 8)
    // rows per thread per step, summed as a small tree before the compensated
    // addition: the same grouping with and without the count, so the fused call's
    // mean equals ce_forward's bit for bit (16 with the targets measured 4-10 us
    // slower at 65536-131072 rows)
    constexpr int U = 8;
    for (int64_t i0 = threadIdx.x; i0 < n; i0 += int64_t(kMeanThreads) * U) {
        float l[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t i = i0 + int64_t(u) * kMeanThreads;
            const bool in = i < n;
            if (!kCounted) ci += (in && target[i] != ignore_idx) ? 1 : 0;
            l[u] = (in && loss_rows) ? loss_rows[i] : 0.f;
        }
#pragma unroll
        for (int w = U / 2; w >= 1; w >>= 1)
#pragma unroll
            for (int u = 0; u < w; ++u) l[u] = l[2 * u] + l[2 * u + 1];
        const float bsum = l[0];
        const float t = fs + bsum;
        if (isfinite(t))  // an infinite or NaN loss propagates through fs alone
            fc += fabsf(fs) >= fabsf(bsum) ? (fs - t) + bsum : (bsum - t) + fs;
        fs = t;
    }
    float hi = fs, lo = 0.f;
    pair_add(hi, lo, fc, 0.f);
    long long c = ci;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        const float h2 = __shfl_xor_sync(0xffffffffu, hi, off), l2 = __shfl_xor_sync(0xffffffffu, lo, off);
        pair_add(hi, lo, h2, l2);
        if (!kCounted) c += __shfl_xor_sync(0xffffffffu, c, off);
    }
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (lane == 0) { sm_h[warp] = hi; sm_l[warp] = lo; sm_c[warp] = c; }
    __syncthreads();
    if (warp == 0) {
        hi = sm_h[lane];
        lo = sm_l[lane];
        c = sm_c[lane];
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            const float h2 = __shfl_xor_sync(0xffffffffu, hi, off), l2 = __shfl_xor_sync(0xffffffffu, lo, off);
            pair_add(hi, lo, h2, l2);
            if (!kCounted) c += __shfl_xor_sync(0xffffffffu, c, off);
        }
        if (kCounted) c = n_valid[0];
        if (lane == 0) {
            // mean: (hi + lo) / N_v with one correction step (0/0 = NaN when every
            // row is ignored); sum: the plain total
            float out;
            if (reduce == VCE_REDUCE_SUM) {
                out = hi + lo;
            } else {
                const float cf = float(c);
                const float q = __fdiv_rn(hi, cf);
                out = isfinite(q) ? q + __fdiv_rn(fmaf(-q, cf, hi) + lo, cf) : q;
            }
            if (loss_out) loss_out[0] = out;
            if (n_valid && !kCounted) n_valid[0] = c;
        }
    }
}

// N_v alone (no loss to reduce): the count of rows whose target is not
// ignore_idx, from integer loads only, sixteen in flight per thread, summed with
// redux.sync per warp and over the warps in shared memory.
constexpr int kCountThreads = 1024;

__global__ void __launch_bounds__(kCountThreads)
count_valid_kernel(const int64_t* __restrict__ target, int64_t n, int64_t ignore_idx, int64_t* __restrict__ n_valid) {
    __shared__ unsigned sm_c[32];
    constexpr int U = 16;
    int ci = 0;  // this thread's count (at most n / 1024 + 16)
    for (int64_t i0 = threadIdx.x; i0 < n; i0 += int64_t(kCountThreads) * U) {
        int64_t t[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t i = i0 + int64_t(u) * kCountThreads;
            t[u] = i < n ? target[i] : ignore_idx;
        }
#pragma unroll
        for (int u = 0; u < U; ++u) ci += t[u] != ignore_idx ? 1 : 0;
    }
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const unsigned wc = __reduce_add_sync(0xffffffffu, unsigned(ci));
    if (lane == 0) sm_c[warp] = wc;
    __syncthreads();
    if (warp == 0) {
        long long c = sm_c[lane];
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) c += __shfl_xor_sync(0xffffffffu, c, off);
        if (lane == 0) n_valid[0] = c;
    }
}

// ---------------------------------------------------------------------------
// token shift for causal language modelling
// ---------------------------------------------------------------------------

// shifted[i] = target[i + 1] unless i is the last position of its sequence of
// ``seq_len`` positions (or of the whole array), where it is ignore_idx.
__global__ void shift_targets_kernel(const int64_t* __restrict__ target, int64_t n, int64_t seq_len,
                                     int64_t ignore_idx, int64_t* __restrict__ shifted) {
    for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
         i += int64_t(gridDim.x) * blockDim.x) {
        const bool last = (i % seq_len == seq_len - 1) || (i == n - 1);
        shifted[i] = last ? ignore_idx : target[i + 1];
    }
}

template <typename T, int THREADS, int MINB>
void fwd_launch(const void* logits, int64_t n_rows, int64_t vocab, int64_t stride,
                const int64_t* target, float eps, int64_t ignore_idx, float* loss_rows,
                float* stats, int* dev_status, cudaStream_t s, int grid) {
    count_launch();
    if (eps != 0.f)
        ce_forward_rows<THREADS, MINB, T, true><<<grid, THREADS, 0, s>>>(
            static_cast<const T*>(logits), n_rows, vocab, stride, target, eps, ignore_idx,
            loss_rows, reinterpret_cast<float2*>(stats), dev_status);
    else
        ce_forward_rows<THREADS, MINB, T, false><<<grid, THREADS, 0, s>>>(
            static_cast<const T*>(logits), n_rows, vocab, stride, target, eps, ignore_idx,
            loss_rows, reinterpret_cast<float2*>(stats), dev_status);
}

template <typename T>
void fwd_dispatch(const void* logits, int64_t n_rows, int64_t vocab, int64_t stride,
                  const int64_t* target, float eps, int64_t ignore_idx, float* loss_rows,
                  float* stats, int* dev_status, cudaStream_t s, int grid) {
    // One CTA per row, threads by row length.  The 128- and 256-thread kernels
    // are held to 32 registers, so 2048 threads (16 or 8 rows) fit on an SM; the
    // 512-thread kernel needs no bound for its 4 rows.  512 threads were measured
    // faster than 1024 for every row above 4096 vectors (0.24 against 0.31 ms at
    // 16384 x 50257 BF16, 0.56 against 0.58 ms at 16384 x 128256).
    const int64_t nvec = vocab / Elem<T>::kVec;
    if (nvec <= 1024)
        fwd_launch<T, 128, 16>(logits, n_rows, vocab, stride, target, eps, ignore_idx, loss_rows, stats, dev_status, s, grid);
    else if (nvec <= 4096)
        fwd_launch<T, 256, 8>(logits, n_rows, vocab, stride, target, eps, ignore_idx, loss_rows, stats, dev_status, s, grid);
    else
        fwd_launch<T, 512, 0>(logits, n_rows, vocab, stride, target, eps, ignore_idx, loss_rows, stats, dev_status, s, grid);
}

template <typename T>
void bwd_dispatch(const void* logits, int64_t n_rows, int64_t vocab, int64_t stride,
                  const int64_t* target, const float* stats, const int64_t* n_valid,
                  const float* grad_output, float eps, int reduce_loss, int64_t ignore_idx,
                  void* dlogits, int* dev_status, cudaStream_t s, int grid) {
    const int64_t nvec = vocab / Elem<T>::kVec;
    const T* z = static_cast<const T*>(logits);
    T* dz = static_cast<T*>(dlogits);
    const float2* st = reinterpret_cast<const float2*>(stats);
    count_launch();
    if (nvec <= 1024)
        ce_backward_rows<128, T><<<grid, 128, 0, s>>>(z, n_rows, vocab, stride, target, st, n_valid,
                                                       grad_output, eps, reduce_loss, ignore_idx, dz, dev_status);
    else if (nvec <= 4096)
        ce_backward_rows<256, T><<<grid, 256, 0, s>>>(z, n_rows, vocab, stride, target, st, n_valid,
                                                       grad_output, eps, reduce_loss, ignore_idx, dz, dev_status);
    else
        ce_backward_rows<512, T><<<grid, 512, 0, s>>>(z, n_rows, vocab, stride, target, st, n_valid,
                                                       grad_output, eps, reduce_loss, ignore_idx, dz, dev_status);
}

// ---------------------------------------------------------------------------
// fused forward + backward (one HBM read, one HBM write per element)
// ---------------------------------------------------------------------------

// Asks L2 to fetch the 16-byte aligned interior of a row from HBM, in 32 KiB
// bulk requests (cp.async.bulk.prefetch.L2).  A hint only: nothing waits on it
// and results do not depend on it; every requested byte lies inside the row.
template <typename T>
__device__ __forceinline__ void prefetch_row_l2(const T* row, int64_t vocab) {
    const uintptr_t b = reinterpret_cast<uintptr_t>(row);
    const uintptr_t a1 = (b + uintptr_t(vocab) * sizeof(T)) & ~uintptr_t(15);
    for (uintptr_t a = (b + 15) & ~uintptr_t(15); a < a1; a += 32768) {
        const uint32_t bytes = uint32_t(a1 - a < 32768 ? a1 - a : 32768);
        asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(a), "r"(bytes) : "memory");
    }
}

// Streams one row through the online (max, sum exp) accumulator.
template <int THREADS, int U, typename T, bool kSmooth>
__device__ __forceinline__ void row_online_lse(const T* p, const RowSplit<T>& sp, int64_t vocab, OnlineLse& acc,
                                               int* st) {
    using E = Elem<T>;
    constexpr int V = E::kVec;
    if (threadIdx.x < sp.head && elem_ok(threadIdx.x, vocab, st)) {
        float v[1] = {E::load1(p + threadIdx.x)};
        acc.push<1, kSmooth>(v);
    }
    const uint4* pv = reinterpret_cast<const uint4*>(p + sp.head);
    int64_t i = threadIdx.x;
    for (; i + (U - 1) * THREADS < sp.nvec; i += U * THREADS) {
        uint4 raw[U];
#pragma unroll
        for (int u = 0; u < U; ++u)  // default caching: the row is read again
            raw[u] = vec_ok(sp, i + u * THREADS, vocab, pv + i + u * THREADS, st) ? pv[i + u * THREADS]
                                                                                  : make_uint4(0, 0, 0, 0);
        push_raw<T, U, kSmooth, true, 2>(acc, raw);
    }
    for (; i < sp.nvec; i += THREADS) {
        float v[V];
        E::unpack(vec_ok(sp, i, vocab, pv + i, st) ? pv[i] : make_uint4(0, 0, 0, 0), v);
        acc.push<V, kSmooth>(v);
    }
    for (int64_t j = sp.tail0 + threadIdx.x; j < vocab; j += THREADS) {
        float v[1] = {elem_ok(j, vocab, st) ? E::load1(p + j) : 0.f};
        acc.push<1, kSmooth>(v);
    }
}

// Row kernel doing the forward and, with the row still in L2, the backward:
// loss, (max, lse) and dlogits = g (softmax - (1-eps) onehot - eps/V) from one
// pass over HBM in each direction.  A persistent grid keeps MINB rows per SM in
// flight, few enough for their second read to hit L2.  With kPrefetch, the CTA
// asks L2 for its next row as its second pass starts, so HBM reads continue
// while the CTA reads L2 and writes gradients (the caller enables it only when
// two rows per CTA fit in L2 with room to spare).
// dlogits may equal logits (the row is overwritten by its gradient).
template <int THREADS, int MINB, int U1, int U2, typename T, bool kSmooth, bool kPrefetch>
__global__ void __launch_bounds__(THREADS, MINB)
ce_fused_rows(const T* logits, int64_t n_rows, int64_t vocab, int64_t stride, const int64_t* __restrict__ target,
              float eps, int64_t ignore_idx, const int64_t* __restrict__ n_valid,
              const float* __restrict__ grad_output, int reduce_loss, float* __restrict__ loss_rows,
              float2* __restrict__ stats, T* dlogits, int* dev_status) {
    using E = Elem<T>;
    constexpr int V = E::kVec;
    constexpr int U = U2;
    __shared__ float sm_part[6 * 32];  // two sets of warp partials (group_merge_all)
    uint32_t set = 0;
    // thread 0: the target element of the last row's gradient, written after the
    // next barrier (see pass 2)
    T* fix_q = nullptr;
    float fix_v = 0.f;
    // the upstream gradient of the mean and sum reductions is the same for every row
    const bool g_rows = reduce_loss == VCE_REDUCE_NONE;
    const float g_all = g_rows ? 0.f : upstream_grad(reduce_loss, grad_output, n_valid, 0);

    for (int64_t row = blockIdx.x; row < n_rows; row += gridDim.x) {
        const int64_t y = target[row];
        const T* p = logits + row * stride;
        T* q = dlogits + row * stride;
        const RowSplit<T> sp(p, vocab);
        if (y == ignore_idx) {
            if (threadIdx.x == 0) {
                loss_rows[row] = 0.f;
                stats[row] = make_float2(0.f, 0.f);
            }
            row_zero<THREADS, T>(q, sp, vocab, dev_status);
            continue;
        }
        const bool bad = y < 0 || y >= vocab;
        // the row's target logit and upstream gradient are requested now and used
        // after the merge, so their latency overlaps the first pass
        const float zy = (threadIdx.x == 0 && !bad) ? E::load1(p + y) : 0.f;
        const float g_row = g_rows ? grad_output[row] : 0.f;
        OnlineLse acc;
        row_online_lse<THREADS, U1, T, kSmooth>(p, sp, vocab, acc, dev_status);
        group_merge_all<THREADS / 32, kSmooth>(acc, sm_part, set, [] { __syncthreads(); });
        set ^= 1u;
        if (threadIdx.x == 0 && fix_q) {  // every thread's stores of that row precede the barrier
            E::store1(fix_q, fix_v);
            fix_q = nullptr;
        }
        const float lse = acc.m + logf(acc.s);
        if (threadIdx.x == 0) {
            float loss;
            if (!bad) {
                loss = lse - zy;
                if (kSmooth) loss = (1.f - eps) * loss + eps * (lse - acc.sum / float(vocab));
            } else {
                loss = __int_as_float(0x7fc00000);
                report(dev_status, VCE_DEVSTATUS_BAD_TARGET);
            }
            loss_rows[row] = loss;
            stats[row] = make_float2(acc.m, lse);
        }
        if (kPrefetch && threadIdx.x == 32) {
            const int64_t next = row + gridDim.x;
            if (next < n_rows && target[next] != ignore_idx) prefetch_row_l2(logits + next * stride, vocab);
        }
        if (bad) {
            row_zero<THREADS, T>(q, sp, vocab, dev_status);
            continue;
        }
        const float g = g_rows ? g_row : g_all;
        const Exp2Offset eo = exp2_offset(lse);
        const float negl = eo.neg;
        const float gp = g * eo.fix;
        const float b = g * eps / float(vocab);
        const float c = g * (1.f - eps);
        // Every element is written as g softmax - g eps / V, with no test for the
        // target in any vector; thread 0 then overwrites the target's element with
        // that value minus g (1 - eps), by the same operations as ce_backward_rows,
        // after the next barrier (the next merge's, or the last one below), which
        // orders it after the store of the thread that wrote the element (2-3%
        // faster on rows of 4096-8000 BF16 elements).
        auto grad1 = [&](int64_t j) {
            if (!elem_ok(j, vocab, dev_status)) return;
            const float z = E::load1(p + j);
            E::store1(q + j, fmaf(gp, ex2f(fmaf(z, kLog2e, negl)), -b));
        };
        if (threadIdx.x < sp.head) grad1(threadIdx.x);
        const uint4* pv = reinterpret_cast<const uint4*>(p + sp.head);
        uint4* qv = reinterpret_cast<uint4*>(q + sp.head);
        auto gradv = [&](const uint4& raw, int64_t i) {
            float v[V];
            E::unpack(raw, v);
            // scalar FMAs here (the same per-lane arithmetic as grad_lanes, so the same
            // bits as ce_backward_rows): the pair form costs this 64-register kernel a spill
#pragma unroll
            for (int k = 0; k < V; ++k) v[k] = fmaf(gp, ex2f(fmaf(v[k], kLog2e, negl)), -b);
            if (vec_ok(sp, i, vocab, qv + i, dev_status)) __stcs(qv + i, E::pack(v));
        };
        int64_t i = threadIdx.x;
        for (; i + (U - 1) * THREADS < sp.nvec; i += U * THREADS) {
            uint4 raw[U];
#pragma unroll
            for (int u = 0; u < U; ++u)
                raw[u] = vec_ok(sp, i + u * THREADS, vocab, pv + i + u * THREADS, dev_status)
                             ? __ldcs(pv + i + u * THREADS) : make_uint4(0, 0, 0, 0);
#pragma unroll
            for (int u = 0; u < U; ++u) gradv(raw[u], i + u * THREADS);
        }
        for (; i < sp.nvec; i += THREADS)
            gradv(vec_ok(sp, i, vocab, pv + i, dev_status) ? __ldcs(pv + i) : make_uint4(0, 0, 0, 0), i);
        for (int64_t j = sp.tail0 + threadIdx.x; j < vocab; j += THREADS) grad1(j);
        if (threadIdx.x == 0 && elem_ok(y, vocab, dev_status)) {
            fix_q = q + y;
            fix_v = __fsub_rn(fmaf(gp, ex2f(fmaf(zy, kLog2e, negl)), -b), c);  // as ce_backward_rows
        }
    }
    __syncthreads();
    if (threadIdx.x == 0 && fix_q) E::store1(fix_q, fix_v);
}

// ---------------------------------------------------------------------------
// fused forward + backward for long rows: rows streamed through a shared-memory
// ring by TMA bulk copies
// ---------------------------------------------------------------------------

// Global -> shared bulk copy (16-byte aligned addresses, size a multiple of 16)
// whose completion is counted on an mbarrier of this CTA.
__device__ __forceinline__ void bulk_load_shared(uint32_t dst, const void* src, uint32_t bytes, uint32_t mbar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                 ::"r"(dst), "l"(src), "r"(bytes), "r"(mbar)
                 : "memory");
}

// The same copy with an L2 eviction-priority hint for the bytes it reads.
__device__ __forceinline__ void bulk_load_shared_hint(uint32_t dst, const void* src, uint32_t bytes, uint32_t mbar,
                                                      uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;"
        ::"r"(dst), "l"(src), "r"(bytes), "r"(mbar), "l"(policy)
        : "memory");
}

__device__ __forceinline__ uint64_t l2_policy_evict_last() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ uint64_t l2_policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// Barrier among the NT compute threads only (the producer warp does not take part).
template <int NT>
__device__ __forceinline__ void compute_sync() {
    asm volatile("bar.sync 1, %0;" ::"n"(NT) : "memory");
}

// group_merge over the compute threads of the cluster kernel (a named barrier
// that leaves the producer warp out); thread 0 ends with the CTA's partial
template <int NT, bool kSum>
__device__ __forceinline__ void compute_merge(OnlineLse& a, float* sm_m, float* sm_s, float* sm_sum) {
    group_merge<NT / 32, kSum>(a, sm_m, sm_s, sm_sum, [] { compute_sync<NT>(); });
}

// NW compute warps, each thread taking PER 16-byte vectors of every full
// chunk; RING_KB KiB of shared memory in equal chunks.
template <int NW, int PER, int RING_KB>
struct RingCfg {
    static constexpr int kThreads = NW * 32;                        // compute threads
    static constexpr uint32_t kChunk = uint32_t(kThreads) * PER * 16;  // bytes per ring slot
    static constexpr int kSlots = int(uint32_t(RING_KB) * 1024 / kChunk);
    // ring, full/empty barriers per slot, two sets of merge partials and the abort
    // flag (the cluster kernel adds its exchange slots and keeps one set)
    static constexpr size_t kSmemBytes = size_t(kSlots) * kChunk + (2 * kSlots) * 8 + (6 * 32 + 2) * 4;
    static_assert(kSlots >= 2 && kSlots <= 16, "ring depth");
};

// Bounded wait that ignores the abort flag (draining copies still in flight:
// they complete on their own, so the long drain limit is never reached in
// practice and the CTA does not exit while a copy into its shared memory runs).
__device__ __forceinline__ bool ring_drain_wait(uint64_t* bar, uint32_t parity) {
    const uint64_t t0 = sm100::globaltimer();
    while (!sm100::mbar_try_wait(bar, parity))
        if (sm100::globaltimer() - t0 > kDrainTimeoutNs) return false;
    return true;
}

// MINB persistent CTAs per SM; warps 0..NW-1 compute, warp NW is the producer.
// The producer's first thread walks the same sequence of rows as the compute
// warps and, for every row that is not ignored, copies the row's 16-byte
// aligned interior into the ring chunk by chunk, once for the first pass and,
// unless the target is out of range, once more for the second pass (the second
// read is served by L2).  It runs ahead of the compute warps by up to the ring
// depth, across the block-wide merge between the passes and across rows, so
// HBM and L2 reads continue while the compute warps merge, and the copies in
// flight (up to the whole ring) take no registers.  The compute warps take
// every chunk in order: pass 1 folds it into the online (max, sum exp), pass 2
// turns it into dlogits written to global memory; the few elements before the
// first 16-byte boundary and after the last are read directly.  With kHint the
// first pass's copies ask L2 to keep the row's lines (evict_last) and the second
// pass's to drop them first (evict_first), so the next row's first-pass reads do
// not push out lines the second pass still needs.
// Every wait is bounded (``timeout_ns``): on timeout the CTA sets its abort
// flag, every role stops waiting, the producer waits for the copies it issued,
// and VCE_DEVSTATUS_TIMEOUT is reported (the outputs are then undefined).
// ``hold`` (failure-detection self-test only) makes the producer issue no copy,
// so the compute warps' first wait runs out with nothing in flight.
template <int NW, int PER, int RING_KB, int MINB, bool kHint, typename T, bool kSmooth>
__global__ void __launch_bounds__(NW * 32 + 32, MINB)
ce_fused_ring(const T* logits, int64_t n_rows, int64_t vocab, int64_t stride, const int64_t* __restrict__ target,
              float eps, int64_t ignore_idx, const int64_t* __restrict__ n_valid,
              const float* __restrict__ grad_output, int reduce_loss, float* __restrict__ loss_rows,
              float2* __restrict__ stats, T* dlogits, int* dev_status, uint64_t timeout_ns, int hold) {
    using E = Elem<T>;
    using C = RingCfg<NW, PER, RING_KB>;
    using namespace sm100;
    constexpr int V = E::kVec;
    constexpr int NT = C::kThreads;
    constexpr uint32_t CH = C::kChunk;
    constexpr int S = C::kSlots;
    extern __shared__ __align__(128) uint8_t smem[];
    uint8_t* ring = smem;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + size_t(S) * CH);
    uint64_t* empty = full + S;
    float* sm_part = reinterpret_cast<float*>(empty + S);  // two sets of warp partials (group_merge_all)
    volatile int* abort_flag = reinterpret_cast<volatile int*>(sm_part + 6 * 32);
    const int tid = threadIdx.x;

    if (tid == 0) {
        for (int i = 0; i < S; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], NW);
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();

    if (tid >= NT) {
        // ---------------- producer ----------------
        if (tid != NT) return;
        uint32_t slot = 0, ph = 0, issued = 0;
        bool ok = true;
        const uint64_t keep = kHint ? l2_policy_evict_last() : 0, drop = kHint ? l2_policy_evict_first() : 0;
        // bounds-checking build: a copy of ``bytes`` from offset ``off`` of a row's
        // 16-byte interior (``total`` bytes from ``src``) into shared memory at
        // ``dst``, which must end by ``dst_end``
        auto copy_ok = [&](const uint8_t* src, uint64_t total, uint64_t off, uint32_t bytes, const uint8_t* dst,
                           const uint8_t* dst_end) {
            return VCE_BOUNDS(aligned16(src + off) && aligned16(dst) && bytes > 0 && bytes % 16 == 0 &&
                                  off + bytes <= total && dst + bytes <= dst_end,
                              dev_status);
        };
        // the next row's target is loaded while this row's copies are issued
        int64_t y_next = int64_t(blockIdx.x) < n_rows ? target[blockIdx.x] : ignore_idx;
        for (int64_t row = blockIdx.x; row < n_rows && ok && !hold; row += gridDim.x) {
            const int64_t y = y_next;
            y_next = row + gridDim.x < n_rows ? target[row + gridDim.x] : ignore_idx;
            if (y == ignore_idx) continue;
            const bool bad = y < 0 || y >= vocab;
            const T* p = logits + row * stride;
            const RowSplit<T> sp(p, vocab);
            const uint64_t total = uint64_t(sp.nvec) * 16;
            const uint8_t* src = reinterpret_cast<const uint8_t*>(p + sp.head);
            for (int pass = 0; pass < (bad ? 1 : 2) && ok; ++pass) {
                for (uint64_t off = 0; off < total; off += CH) {
                    if (!mbar_wait(&empty[slot], ph ^ 1, abort_flag, timeout_ns)) {
                        ok = false;
                        break;
                    }
                    const uint32_t bytes = uint32_t(total - off < CH ? total - off : CH);
                    const bool cok = copy_ok(src, total, off, bytes, ring + size_t(slot) * CH,
                                             ring + size_t(slot + 1) * CH);
                    mbar_arrive_expect_tx(&full[slot], cok ? bytes : 0u);
                    if (cok && kHint)
                        bulk_load_shared_hint(smem_u32(ring + size_t(slot) * CH), src + off, bytes,
                                              smem_u32(&full[slot]), pass == 0 ? keep : drop);
                    else if (cok)
                        bulk_load_shared(smem_u32(ring + size_t(slot) * CH), src + off, bytes,
                                         smem_u32(&full[slot]));
                    ++issued;
                    if (++slot == uint32_t(S)) {
                        slot = 0;
                        ph ^= 1;
                    }
                }
            }
        }
        // wait for the last copy into every slot that received one (all of them
        // have completed already unless the CTA gave up)
        for (uint32_t i = 0; i < uint32_t(S) && i < issued; ++i) {
            const uint32_t last = i + ((issued - 1 - i) / S) * S;
            ring_drain_wait(&full[i], (last / S) & 1);
        }
        if (!ok || *abort_flag) report(dev_status, VCE_DEVSTATUS_TIMEOUT);
        return;
    }

    // ---------------- compute warps ----------------
    // The scalars of a row (its target, its head and tail elements outside the
    // copied interior, its target logit and, without reduction, its upstream
    // gradient) are fetched one row ahead: the next row's target is loaded as a
    // row starts, and once the first pass has given it time to arrive, the
    // next row's other scalars are loaded, so no dependent global load stands
    // between a row's chunks, its merge and its second pass.  Ignored rows are
    // still never read, and every value enters the arithmetic in the same
    // order as before (the head first, the tail last).
    const int lane = tid & 31;
    uint32_t slot = 0, ph = 0;
    uint32_t set = 0;  // merge partial set (group_merge_all)
    bool ok = true;
    // wait for the next chunk; false once this CTA has given up
    auto take = [&]() -> bool {
        if (ok && !mbar_wait(&full[slot], ph, abort_flag, timeout_ns)) ok = false;
        return ok;
    };
    auto release = [&]() {
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[slot]);
        if (++slot == uint32_t(S)) {
            slot = 0;
            ph ^= 1;
        }
    };
    const bool g_rows = reduce_loss == VCE_REDUCE_NONE;
    const float g_all = g_rows ? 0.f : upstream_grad(reduce_loss, grad_output, n_valid, 0);
    struct Scalars {
        float zh = 0.f, zt = 0.f, zy = 0.f, g = 0.f;  // head element, tail element, target logit, gradient
    };
    // loads the scalars of a row that is not ignored (each thread those it uses)
    auto fetch = [&](int64_t r, int64_t yr) {
        Scalars sc;
        const T* pr = logits + r * stride;
        const RowSplit<T> spr(pr, vocab);
        if (tid < spr.head && elem_ok(tid, vocab, dev_status)) sc.zh = E::load1(pr + tid);
        if (spr.tail0 + tid < vocab && elem_ok(spr.tail0 + tid, vocab, dev_status))
            sc.zt = E::load1(pr + spr.tail0 + tid);  // the tail is shorter than a vector
        if (tid == 0 && yr >= 0 && yr < vocab) sc.zy = E::load1(pr + yr);
        if (g_rows) sc.g = grad_output[r];
        return sc;
    };
    int64_t y = 0;
    Scalars cur;
    if (int64_t(blockIdx.x) < n_rows) {
        y = target[blockIdx.x];
        if (y != ignore_idx) cur = fetch(blockIdx.x, y);
    }
    for (int64_t row = blockIdx.x; row < n_rows; row += gridDim.x) {
        const int64_t nrow = row + gridDim.x;
        const int64_t ny = nrow < n_rows ? target[nrow] : ignore_idx;  // used after this row's first pass
        const T* p = logits + row * stride;
        T* q = dlogits + row * stride;
        const RowSplit<T> sp(p, vocab);
        if (y == ignore_idx) {
            if (tid == 0) {
                loss_rows[row] = 0.f;
                stats[row] = make_float2(0.f, 0.f);
            }
            row_zero<NT, T>(q, sp, vocab, dev_status);
            cur = ny != ignore_idx ? fetch(nrow, ny) : Scalars();
            y = ny;
            continue;
        }
        const bool bad = y < 0 || y >= vocab;
        const uint64_t total = uint64_t(sp.nvec) * 16;

        // pass 1: online (max, sum exp) and sum of logits
        OnlineLse acc;
        if (tid < sp.head) {
            float v[1] = {cur.zh};
            acc.push<1, kSmooth>(v);
        }
        for (uint64_t off = 0; off < total; off += CH) {
            if (take()) {
                const uint4* src = reinterpret_cast<const uint4*>(ring + size_t(slot) * CH);
                if (total - off >= CH) {
                    uint4 raw[PER];
#pragma unroll
                    for (int u = 0; u < PER; ++u) raw[u] = src[tid + u * NT];
#pragma unroll
                    for (int u = 0; u < PER; ++u) {
                        float v[V];
                        E::unpack(raw[u], v);
                        acc.push<V, kSmooth>(v);
                    }
                } else {
                    const uint32_t nv = uint32_t(total - off) / 16;
                    for (uint32_t j = tid; j < nv; j += NT) {
                        float v[V];
                        E::unpack(src[j], v);
                        acc.push<V, kSmooth>(v);
                    }
                }
            }
            release();
        }
        if (sp.tail0 + tid < vocab) {
            float v[1] = {cur.zt};
            acc.push<1, kSmooth>(v);
        }
        group_merge_all<NW, kSmooth>(acc, sm_part, set, [] { compute_sync<NT>(); });
        set ^= 1u;
        const float lse = acc.m + logf(acc.s);
        if (tid == 0) {
            float loss;
            if (!bad) {
                loss = lse - cur.zy;
                if (kSmooth) loss = (1.f - eps) * loss + eps * (lse - acc.sum / float(vocab));
            } else {
                loss = __int_as_float(0x7fc00000);
                report(dev_status, VCE_DEVSTATUS_BAD_TARGET);
            }
            loss_rows[row] = loss;
            stats[row] = make_float2(acc.m, lse);
        }
        // the next row's target has arrived during the first pass: fetch its
        // other scalars now, to arrive during this row's second pass
        const Scalars nxt = ny != ignore_idx ? fetch(nrow, ny) : Scalars();
        if (bad) {
            row_zero<NT, T>(q, sp, vocab, dev_status);
            cur = nxt;
            y = ny;
            continue;
        }

        // pass 2: dlogits = g (softmax - (1 - eps) onehot - eps / V).  (Writing
        // the target's element apart, after the next barrier, as the short-row
        // kernel does, measured 7% faster or slower here depending on the row
        // length, about even overall, so each vector tests for the target.)
        const float g = g_rows ? cur.g : g_all;
        const Exp2Offset eo = exp2_offset(lse);
        const float negl = eo.neg;
        const float gp = g * eo.fix;
        const float b = g * eps / float(vocab);
        const float c = g * (1.f - eps);
        auto grad1 = [&](int64_t j, float z) {
            float d = fmaf(gp, ex2f(fmaf(z, kLog2e, negl)), -b);
            if (j == y) d = __fsub_rn(d, c);
            if (elem_ok(j, vocab, dev_status)) E::store1(q + j, d);
        };
        if (tid < sp.head) grad1(tid, cur.zh);
        uint4* qv = reinterpret_cast<uint4*>(q + sp.head);
        auto gradv = [&](const uint4& raw, int64_t i) {
            float v[V];
            E::unpack(raw, v);
            grad_lanes<V>(v, gp, negl, b);
            const int64_t base = sp.head + i * V;
            if (uint64_t(y - base) < uint64_t(V)) {
#pragma unroll
                for (int k = 0; k < V; ++k) v[k] = __fsub_rn(v[k], (base + k == y) ? c : 0.f);
            }
            if (vec_ok(sp, i, vocab, qv + i, dev_status)) __stcs(qv + i, E::pack(v));
        };
        for (uint64_t off = 0; off < total; off += CH) {
            if (take()) {
                const uint4* src = reinterpret_cast<const uint4*>(ring + size_t(slot) * CH);
                const int64_t i0 = int64_t(off / 16);
                if (total - off >= CH) {
                    uint4 raw[PER];
#pragma unroll
                    for (int u = 0; u < PER; ++u) raw[u] = src[tid + u * NT];
#pragma unroll
                    for (int u = 0; u < PER; ++u) gradv(raw[u], i0 + tid + u * NT);
                } else {
                    const uint32_t nv = uint32_t(total - off) / 16;
                    for (uint32_t j = tid; j < nv; j += NT) gradv(src[j], i0 + j);
                }
            }
            release();
        }
        if (sp.tail0 + tid < vocab) grad1(sp.tail0 + tid, cur.zt);
        cur = nxt;
        y = ny;
    }
    // a compute thread whose wait gave up reports it too: the producer may have
    // issued its last copy and returned before the CTA gave up
    if (!ok) report(dev_status, VCE_DEVSTATUS_TIMEOUT);
}

// Rows whose two passes would keep too much of L2 busy when one SM takes the
// whole row (BF16 rows above 448 KiB, FP32 above 400 KiB: 152 such rows in
// flight hold 60-70 MB or more of lines between their first and second reads,
// and the second pass starts to miss): the two CTAs of a cluster (two SMs)
// split every row they take.  Rank 0 owns the
// first half of the row's interior chunks and the head elements before it,
// rank 1 the rest and the tail elements, so each SM keeps only half a row in
// L2 between the passes.  Each CTA runs the ring kernel's producer and compute
// warps over its half.  After the first pass each CTA merges its own partial
// (max, sum of exp, sum of logits), sends it to the peer's shared memory
// (st.shared::cluster, then a release-arrive on the peer's mbarrier), waits
// for the peer's (bounded, acquire at cluster scope) and merges the two in
// rank order, so both CTAs hold the same lse; rank 0 writes the loss and the
// statistics.  The exchange uses two slots by row parity: a CTA writes slot
// b for row k only after it received the peer's row k-1 partial, which the
// peer sent after reading slot b for row k-2.  Every thread of both CTAs meets
// at a cluster barrier before exiting, so no CTA leaves while its peer may
// still write into its shared memory.  Waits are bounded as in the ring
// kernel; ``hold`` (self-test) stops the producers' copies.
template <int NW, int PER, int RING_KB, bool kHint, typename T, bool kSmooth>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(NW * 32 + 32, 1)
ce_fused_ring_pair(const T* logits, int64_t n_rows, int64_t vocab, int64_t stride,
                   const int64_t* __restrict__ target, float eps, int64_t ignore_idx,
                   const int64_t* __restrict__ n_valid, const float* __restrict__ grad_output, int reduce_loss,
                   float* __restrict__ loss_rows, float2* __restrict__ stats, T* dlogits, int* dev_status,
                   uint64_t timeout_ns, int hold) {
    using E = Elem<T>;
    using C = RingCfg<NW, PER, RING_KB>;
    using namespace sm100;
    constexpr int V = E::kVec;
    constexpr int NT = C::kThreads;
    constexpr uint32_t CH = C::kChunk;
    constexpr int S = C::kSlots;
    extern __shared__ __align__(128) uint8_t smem[];
    uint8_t* ring = smem;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + size_t(S) * CH);
    uint64_t* empty = full + S;
    uint64_t* xbar = empty + S;                        // [2] the peer's partial has arrived (by row parity)
    float* xval = reinterpret_cast<float*>(xbar + 2);  // [2][4] the peer's (max, sum exp, sum z)
    float* sm_m = xval + 8;
    float* sm_s = sm_m + 32;
    float* sm_sum = sm_s + 32;
    float* sm_lse = sm_sum + 32;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(sm_lse + 1);
    const int tid = threadIdx.x;
    const uint32_t rank = cluster_ctarank();
    const int64_t cid = blockIdx.x / 2, ncl = gridDim.x / 2;

    if (tid == 0) {
        for (int i = 0; i < S; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], NW);
        }
        mbar_init(&xbar[0], 1);
        mbar_init(&xbar[1], 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    cluster_sync();  // both CTAs' exchange barriers exist before either arrives on the other's

    // this CTA's share [lo, hi) of a row's 16-byte interior of ``total`` bytes
    auto share = [&](uint64_t total, uint64_t& lo, uint64_t& hi) {
        const uint64_t nch = (total + CH - 1) / CH, half = (nch + 1) / 2 * CH;
        const uint64_t mid = half < total ? half : total;
        lo = rank == 0 ? 0 : mid;
        hi = rank == 0 ? mid : total;
    };

    if (tid >= NT) {
        if (tid == NT) {
            // ---------------- producer (this CTA's share of every row) ----------------
            uint32_t slot = 0, ph = 0, issued = 0;
            bool ok = true;
            const uint64_t keep = kHint ? l2_policy_evict_last() : 0, drop = kHint ? l2_policy_evict_first() : 0;
            auto copy_ok = [&](const uint8_t* src, uint64_t off, uint32_t bytes, uint64_t hi, const uint8_t* dst) {
                return VCE_BOUNDS(aligned16(src + off) && aligned16(dst) && bytes > 0 && bytes % 16 == 0 &&
                                      off + bytes <= hi && dst + bytes <= ring + size_t(S) * CH,
                                  dev_status);
            };
            int64_t y_next = cid < n_rows ? target[cid] : ignore_idx;
            for (int64_t row = cid; row < n_rows && ok && !hold; row += ncl) {
                const int64_t y = y_next;
                y_next = row + ncl < n_rows ? target[row + ncl] : ignore_idx;
                if (y == ignore_idx) continue;
                const bool bad = y < 0 || y >= vocab;
                const T* p = logits + row * stride;
                const RowSplit<T> sp(p, vocab);
                uint64_t lo, hi;
                share(uint64_t(sp.nvec) * 16, lo, hi);
                const uint8_t* src = reinterpret_cast<const uint8_t*>(p + sp.head);
                for (int pass = 0; pass < (bad ? 1 : 2) && ok; ++pass) {
                    for (uint64_t off = lo; off < hi; off += CH) {
                        if (!mbar_wait(&empty[slot], ph ^ 1, abort_flag, timeout_ns)) {
                            ok = false;
                            break;
                        }
                        const uint32_t bytes = uint32_t(hi - off < CH ? hi - off : CH);
                        uint8_t* dst = ring + size_t(slot) * CH;
                        const bool cok = copy_ok(src, off, bytes, hi, dst);
                        mbar_arrive_expect_tx(&full[slot], cok ? bytes : 0u);
                        if (cok && kHint)
                            bulk_load_shared_hint(smem_u32(dst), src + off, bytes, smem_u32(&full[slot]),
                                                  pass == 0 ? keep : drop);
                        else if (cok)
                            bulk_load_shared(smem_u32(dst), src + off, bytes, smem_u32(&full[slot]));
                        ++issued;
                        if (++slot == uint32_t(S)) {
                            slot = 0;
                            ph ^= 1;
                        }
                    }
                }
            }
            for (uint32_t i = 0; i < uint32_t(S) && i < issued; ++i) {
                const uint32_t last = i + ((issued - 1 - i) / S) * S;
                ring_drain_wait(&full[i], (last / S) & 1);
            }
            if (!ok || *abort_flag) report(dev_status, VCE_DEVSTATUS_TIMEOUT);
        }
    } else {
        // ---------------- compute warps (this CTA's share of every row) ----------------
        const int lane = tid & 31;
        uint32_t slot = 0, ph = 0, xk = 0;  // xk: rows whose partials were exchanged so far
        bool ok = true;
        auto take = [&]() -> bool {
            if (ok && !mbar_wait(&full[slot], ph, abort_flag, timeout_ns)) ok = false;
            return ok;
        };
        auto release = [&]() {
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[slot]);
            if (++slot == uint32_t(S)) {
                slot = 0;
                ph ^= 1;
            }
        };
        const bool g_rows = reduce_loss == VCE_REDUCE_NONE;
        const float g_all = g_rows ? 0.f : upstream_grad(reduce_loss, grad_output, n_valid, 0);
        struct Scalars {
            float zh = 0.f, zt = 0.f, zy = 0.f, g = 0.f;
        };
        // the next row's scalars, fetched a row ahead as in the ring kernel: rank 0
        // owns the head elements and the loss (target logit), rank 1 the tail
        auto fetch = [&](int64_t r, int64_t yr) {
            Scalars sc;
            const T* pr = logits + r * stride;
            const RowSplit<T> spr(pr, vocab);
            if (rank == 0 && tid < spr.head && elem_ok(tid, vocab, dev_status)) sc.zh = E::load1(pr + tid);
            if (rank == 1 && spr.tail0 + tid < vocab && elem_ok(spr.tail0 + tid, vocab, dev_status))
                sc.zt = E::load1(pr + spr.tail0 + tid);
            if (rank == 0 && tid == 0 && yr >= 0 && yr < vocab) sc.zy = E::load1(pr + yr);
            if (g_rows) sc.g = grad_output[r];
            return sc;
        };
        int64_t y = 0;
        Scalars cur;
        if (cid < n_rows) {
            y = target[cid];
            if (y != ignore_idx) cur = fetch(cid, y);
        }
        for (int64_t row = cid; row < n_rows; row += ncl) {
            const int64_t nrow = row + ncl;
            const int64_t ny = nrow < n_rows ? target[nrow] : ignore_idx;
            const T* p = logits + row * stride;
            T* q = dlogits + row * stride;
            const RowSplit<T> sp(p, vocab);
            uint64_t lo, hi;
            share(uint64_t(sp.nvec) * 16, lo, hi);
            if (y == ignore_idx) {
                if (rank == 0 && tid == 0) {
                    loss_rows[row] = 0.f;
                    stats[row] = make_float2(0.f, 0.f);
                }
                part_zero<NT, T>(q, sp, vocab, int64_t(lo / 16), int64_t(hi / 16), rank == 0, rank == 1, dev_status);
                cur = ny != ignore_idx ? fetch(nrow, ny) : Scalars();
                y = ny;
                continue;
            }
            const bool bad = y < 0 || y >= vocab;

            // pass 1 over this CTA's share
            OnlineLse acc;
            if (rank == 0 && tid < sp.head) {
                float v[1] = {cur.zh};
                acc.push<1, kSmooth>(v);
            }
            for (uint64_t off = lo; off < hi; off += CH) {
                if (take()) {
                    const uint4* src = reinterpret_cast<const uint4*>(ring + size_t(slot) * CH);
                    if (hi - off >= CH) {
                        uint4 raw[PER];
#pragma unroll
                        for (int u = 0; u < PER; ++u) raw[u] = src[tid + u * NT];
#pragma unroll
                        for (int u = 0; u < PER; ++u) {
                            float v[V];
                            E::unpack(raw[u], v);
                            acc.push<V, kSmooth>(v);
                        }
                    } else {
                        const uint32_t nv = uint32_t(hi - off) / 16;
                        for (uint32_t j = tid; j < nv; j += NT) {
                            float v[V];
                            E::unpack(src[j], v);
                            acc.push<V, kSmooth>(v);
                        }
                    }
                }
                release();
            }
            if (rank == 1 && sp.tail0 + tid < vocab) {
                float v[1] = {cur.zt};
                acc.push<1, kSmooth>(v);
            }
            compute_merge<NT, kSmooth>(acc, sm_m, sm_s, sm_sum);  // thread 0: this CTA's partial
            if (tid == 0) {
                // exchange the partials with the peer CTA, then merge them in rank order
                const uint32_t b = xk & 1u;
                const uint32_t peer = rank ^ 1u;
                const uint32_t pv = mapa_shared(smem_u32(&xval[b * 4]), peer);
                st_shared_cluster(pv, __float_as_int(acc.m));
                st_shared_cluster(pv + 4, __float_as_int(acc.s));
                st_shared_cluster(pv + 8, __float_as_int(acc.sum));
                mbar_arrive_cluster(mapa_shared(smem_u32(&xbar[b]), peer));
                if (ok && !mbar_wait<true>(&xbar[b], (xk >> 1) & 1u, abort_flag, timeout_ns)) ok = false;
                OnlineLse other;
                other.m = xval[b * 4];
                other.s = xval[b * 4 + 1];
                other.sum = xval[b * 4 + 2];
                OnlineLse t = rank == 0 ? acc : other;
                const OnlineLse& u = rank == 0 ? other : acc;
                t.merge(u.m, u.s, u.sum);
                const float lse = t.m + logf(t.s);
                if (rank == 0) {
                    float loss;
                    if (!bad) {
                        loss = lse - cur.zy;
                        if (kSmooth) loss = (1.f - eps) * loss + eps * (lse - t.sum / float(vocab));
                    } else {
                        loss = __int_as_float(0x7fc00000);
                        report(dev_status, VCE_DEVSTATUS_BAD_TARGET);
                    }
                    loss_rows[row] = loss;
                    stats[row] = make_float2(t.m, lse);
                }
                *sm_lse = lse;
            }
            ++xk;
            compute_sync<NT>();
            const Scalars nxt = ny != ignore_idx ? fetch(nrow, ny) : Scalars();
            if (bad) {
                part_zero<NT, T>(q, sp, vocab, int64_t(lo / 16), int64_t(hi / 16), rank == 0, rank == 1, dev_status);
                cur = nxt;
                y = ny;
                continue;
            }

            // pass 2 over this CTA's share: dlogits = g (softmax - (1 - eps) onehot - eps / V)
            const float g = g_rows ? cur.g : g_all;
            const Exp2Offset eo = exp2_offset(*sm_lse);
            const float negl = eo.neg;
            const float gp = g * eo.fix;
            const float bsh = g * eps / float(vocab);
            const float c = g * (1.f - eps);
            auto grad1 = [&](int64_t j, float z) {
                float d = fmaf(gp, ex2f(fmaf(z, kLog2e, negl)), -bsh);
                if (j == y) d = __fsub_rn(d, c);
                if (elem_ok(j, vocab, dev_status)) E::store1(q + j, d);
            };
            if (rank == 0 && tid < sp.head) grad1(tid, cur.zh);
            uint4* qv = reinterpret_cast<uint4*>(q + sp.head);
            auto gradv = [&](const uint4& raw, int64_t i) {
                float v[V];
                E::unpack(raw, v);
                grad_lanes<V>(v, gp, negl, bsh);
                const int64_t base = sp.head + i * V;
                if (uint64_t(y - base) < uint64_t(V)) {
#pragma unroll
                    for (int k = 0; k < V; ++k) v[k] = __fsub_rn(v[k], (base + k == y) ? c : 0.f);
                }
                if (vec_ok(sp, i, vocab, qv + i, dev_status)) __stcs(qv + i, E::pack(v));
            };
            for (uint64_t off = lo; off < hi; off += CH) {
                if (take()) {
                    const uint4* src = reinterpret_cast<const uint4*>(ring + size_t(slot) * CH);
                    const int64_t i0 = int64_t(off / 16);
                    if (hi - off >= CH) {
                        uint4 raw[PER];
#pragma unroll
                        for (int u = 0; u < PER; ++u) raw[u] = src[tid + u * NT];
#pragma unroll
                        for (int u = 0; u < PER; ++u) gradv(raw[u], i0 + tid + u * NT);
                    } else {
                        const uint32_t nv = uint32_t(hi - off) / 16;
                        for (uint32_t j = tid; j < nv; j += NT) gradv(src[j], i0 + j);
                    }
                }
                release();
            }
            if (rank == 1 && sp.tail0 + tid < vocab) grad1(sp.tail0 + tid, cur.zt);
            cur = nxt;
            y = ny;
        }
        if (!ok) report(dev_status, VCE_DEVSTATUS_TIMEOUT);
    }
    __syncwarp();
    cluster_sync();  // the peer no longer writes into this CTA's shared memory
}

template <typename T, int NW, int PER, int RING_KB, bool kHint>
void pair_launch(const void* logits, int64_t n_rows, int64_t vocab, int64_t stride, const int64_t* target,
                 float eps, int64_t ignore_idx, const int64_t* n_valid, const float* grad_output, int reduce_loss,
                 float* loss_rows, float* stats, void* dlogits, int* dev_status, cudaStream_t s,
                 const DeviceInfo& dev, const PipeDiag& diag) {
    using C = RingCfg<NW, PER, RING_KB>;
    constexpr size_t kSmem = C::kSmemBytes + 64;  // two exchange barriers and slots beyond the ring's layout
    auto kern = eps != 0.f ? ce_fused_ring_pair<NW, PER, RING_KB, kHint, T, true>
                           : ce_fused_ring_pair<NW, PER, RING_KB, kHint, T, false>;
    static std::mutex mu;
    static bool raised[2][64] = {};
    const int k = eps != 0.f ? 1 : 0;
    {
        std::lock_guard<std::mutex> lock(mu);
        if (!raised[k][dev.ordinal]) {
            if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(kSmem)) != cudaSuccess)
                return;  // not launched: the caller's cudaGetLastError() reports the failure
            raised[k][dev.ordinal] = true;
        }
    }
    const int64_t pairs = dev.num_sms / 2;
    const int grid = int(2 * (n_rows < pairs ? n_rows : pairs));  // a cluster of two CTAs per row in flight
    count_launch();
    kern<<<grid, C::kThreads + 32, kSmem, s>>>(
        static_cast<const T*>(logits), n_rows, vocab, stride, target, eps, ignore_idx, n_valid, grad_output,
        reduce_loss, loss_rows, reinterpret_cast<float2*>(stats), static_cast<T*>(dlogits), dev_status,
        diag.timeout_ns, diag.hold);
}

template <typename T, int NW, int PER, int RING_KB, int MINB, bool kHint>
void ring_launch(const void* logits, int64_t n_rows, int64_t vocab, int64_t stride, const int64_t* target,
                 float eps, int64_t ignore_idx, const int64_t* n_valid, const float* grad_output, int reduce_loss,
                 float* loss_rows, float* stats, void* dlogits, int* dev_status, cudaStream_t s,
                 const DeviceInfo& dev, const PipeDiag& diag) {
    using C = RingCfg<NW, PER, RING_KB>;
    auto kern = eps != 0.f ? ce_fused_ring<NW, PER, RING_KB, MINB, kHint, T, true>
                           : ce_fused_ring<NW, PER, RING_KB, MINB, kHint, T, false>;
    // the dynamic shared-memory limit is a per-device attribute of each kernel
    static std::mutex mu;
    static bool raised[2][64] = {};
    const int k = eps != 0.f ? 1 : 0;
    {
        std::lock_guard<std::mutex> lock(mu);
        if (!raised[k][dev.ordinal]) {
            if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(C::kSmemBytes)) !=
                cudaSuccess)
                return;  // not launched: the caller's cudaGetLastError() reports the failure
            raised[k][dev.ordinal] = true;
        }
    }
    const int64_t cap = int64_t(dev.num_sms) * MINB;
    const int grid = int(n_rows < cap ? n_rows : cap);
    count_launch();
    kern<<<grid, C::kThreads + 32, C::kSmemBytes, s>>>(
        static_cast<const T*>(logits), n_rows, vocab, stride, target, eps, ignore_idx, n_valid, grad_output,
        reduce_loss, loss_rows, reinterpret_cast<float2*>(stats), static_cast<T*>(dlogits), dev_status,
        diag.timeout_ns, diag.hold);
}

template <typename T, int THREADS, int MINB, int U1, int U2, bool kPrefetch>
void fused_launch(const void* logits, int64_t n_rows, int64_t vocab, int64_t stride, const int64_t* target,
                  float eps, int64_t ignore_idx, const int64_t* n_valid, const float* grad_output,
                  int reduce_loss, float* loss_rows, float* stats, void* dlogits, int* dev_status,
                  cudaStream_t s, int grid) {
    const T* z = static_cast<const T*>(logits);
    T* dz = static_cast<T*>(dlogits);
    float2* st = reinterpret_cast<float2*>(stats);
    count_launch();
    if (eps != 0.f)
        ce_fused_rows<THREADS, MINB, U1, U2, T, true, kPrefetch><<<grid, THREADS, 0, s>>>(
            z, n_rows, vocab, stride, target, eps, ignore_idx, n_valid, grad_output, reduce_loss, loss_rows, st,
            dz, dev_status);
    else
        ce_fused_rows<THREADS, MINB, U1, U2, T, false, kPrefetch><<<grid, THREADS, 0, s>>>(
            z, n_rows, vocab, stride, target, eps, ignore_idx, n_valid, grad_output, reduce_loss, loss_rows, st,
            dz, dev_status);
}

// Persistent grid of ``per_sm`` CTAs per SM, or one CTA per row if fewer.
inline int fused_grid(int64_t n_rows, int num_sms, int per_sm) {
    const int64_t cap = int64_t(num_sms) * per_sm;
    return int(n_rows < cap ? n_rows : cap);
}

template <typename T>
void fused_dispatch(const void* logits, int64_t n_rows, int64_t vocab, int64_t stride, const int64_t* target,
                    float eps, int64_t ignore_idx, const int64_t* n_valid, const float* grad_output,
                    int reduce_loss, float* loss_rows, float* stats, void* dlogits, int* dev_status,
                    cudaStream_t s, const DeviceInfo& dev, const PipeDiag& diag) {
    // Rows up to 1024 vectors (16 KiB): 128 threads per row, 8 CTAs per SM, and
    // the next-row L2 prefetch while two rows per CTA take at most two thirds of
    // L2.  Longer rows: the TMA-fed ring kernel, shaped by row length and element
    // size (an FP32 row carries half the arithmetic per byte of a BF16 row, so it
    // favours fewer, larger CTAs).  Each compute thread takes PER 16-byte vectors
    // of every chunk: more vectors between two waits on the ring give it more
    // independent arithmetic to interleave, which the latency-bound short and mid
    // rows need.  Measured at 16384 rows, fraction of the copy peak (in brackets
    // the same ring with 4 vectors per thread):
    //   BF16 up to 44 KiB: four CTAs per SM, 4 compute warps x 8 vectors, 48 KiB
    //     rings of three chunks (V = 10000: 0.72; 13000: 0.79; 16000: 0.85;
    //     22500: 0.87 [0.70-0.87]);
    //   BF16 up to 88 KiB: two CTAs per SM, 8 compute warps x 7 vectors, 112 KiB
    //     rings of four 28 KiB chunks (25000: 0.86; 32000: 0.90; 35000: 0.90;
    //     38000: 0.92; 44500: 0.92 [0.82-0.92]);
    //   BF16 up to 112 KiB: two CTAs per SM, 8 compute warps x 8 vectors, 96 KiB
    //     rings of three chunks (47000: 0.93; 50257: 0.92; 55000: 0.925
    //     [0.91-0.93]);
    //   BF16 up to 240 KiB: one CTA per SM, 16 compute warps x 4 vectors, a 224
    //     KiB ring and L2 hints that keep the first pass's bytes for the second
    //     (65536: 0.95; 100352: 0.97; 120000: 0.96; the 192 KiB ring 0.94);
    //   BF16 up to 288 KiB: the same with a 192 KiB ring (128256: 0.97-0.98;
    //     140000: 0.96; 8 vectors per thread 0.94-0.97);
    //   BF16 up to 448 KiB: the 192 KiB ring with 8 vectors per thread, in three
    //     64 KiB chunks (160000: 0.95; 180000: 0.94; 205000: 0.90; 210000: 0.87
    //     [0.83-0.92]);
    //   FP32 up to 56 KiB: two CTAs per SM, 8 compute warps x 8 vectors, 96 KiB
    //     rings (V = 7000: 0.85; 10000: 0.90; 13500: 0.87 [0.81-0.87]);
    //   FP32 up to 128 KiB: one CTA per SM, 16 compute warps x 4 vectors, the 192
    //     KiB ring with L2 hints (16000: 0.91; 25000: 0.96);
    //   FP32 up to 400 KiB: the same with 8 vectors per thread (50257: 0.96;
    //     95000: 0.885; 102000: 0.88 [0.86-0.95]);
    //   longer: each row split between the two CTAs of a cluster (two SMs),
    //     each with the 192 KiB ring (4 vectors per thread) over its half, so
    //     each SM keeps half a row in L2 between the passes (BF16 256000: 0.90
    //     against 0.81 for the single-CTA ring; FP32 128256: 0.92 against 0.83).
    //     On shorter rows the exchange of the halves' partials costs more than it
    //     saves (BF16 205000: 0.82 against 0.90; FP32 102000: 0.86 against 0.88),
    //     and the pair with 6-8 vectors per thread splits rows into uneven halves
    //     of whole chunks (0.77-0.87).
    // (Over ring shapes of 4-16 compute warps, 2-8 vectors per thread, 8-64 KiB
    // chunks, 48-224 KiB rings and 1-4 CTAs per SM.)  Where a ring has as many
    // compute threads as the forward kernel has threads per row, every thread
    // takes the same vectors in the same order, whatever its chunk size, so those
    // rows equal ce_forward + ce_backward bit for bit: BF16 rows of 48-64 KiB and
    // FP32 rows of 16-56 KiB (8 warps, the forward's 256 threads), and rows of
    // 112-448 KiB BF16 or 64-400 KiB FP32 (16 warps, its 512), as the rows up to
    // 16 KiB do.
    const int64_t nvec = vocab / Elem<T>::kVec;
    const int64_t bytes = nvec * 16;
    const double l2 = double(dev.l2_bytes), row = double(vocab) * double(sizeof(T));
#define VCE_FUSED_ARGS logits, n_rows, vocab, stride, target, eps, ignore_idx, n_valid, grad_output, reduce_loss, \
                       loss_rows, stats, dlogits, dev_status, s
    constexpr int64_t KiB = 1024;
    if (nvec <= 1024) {
        const int grid = fused_grid(n_rows, dev.num_sms, 8);
        if (double(grid) * 2 * row <= l2 * 2.0 / 3.0) fused_launch<T, 128, 8, 4, 2, true>(VCE_FUSED_ARGS, grid);
        else fused_launch<T, 128, 8, 4, 2, false>(VCE_FUSED_ARGS, grid);
    } else if (bytes > (sizeof(T) == 4 ? 400 : 448) * KiB) {
        pair_launch<T, 16, 4, 192, true>(VCE_FUSED_ARGS, dev, diag);
    } else if constexpr (sizeof(T) == 4) {
        if (bytes <= 56 * KiB) ring_launch<T, 8, 8, 96, 2, false>(VCE_FUSED_ARGS, dev, diag);
        else if (bytes <= 128 * KiB) ring_launch<T, 16, 4, 192, 1, true>(VCE_FUSED_ARGS, dev, diag);
        else ring_launch<T, 16, 8, 192, 1, true>(VCE_FUSED_ARGS, dev, diag);
    } else {
        if (bytes <= 44 * KiB) ring_launch<T, 4, 8, 48, 4, false>(VCE_FUSED_ARGS, dev, diag);
        else if (bytes <= 88 * KiB) ring_launch<T, 8, 7, 112, 2, false>(VCE_FUSED_ARGS, dev, diag);
        else if (bytes <= 112 * KiB) ring_launch<T, 8, 8, 96, 2, false>(VCE_FUSED_ARGS, dev, diag);
        else if (bytes <= 240 * KiB) ring_launch<T, 16, 4, 224, 1, true>(VCE_FUSED_ARGS, dev, diag);
        else if (bytes <= 288 * KiB) ring_launch<T, 16, 4, 192, 1, true>(VCE_FUSED_ARGS, dev, diag);
        else ring_launch<T, 16, 8, 192, 1, true>(VCE_FUSED_ARGS, dev, diag);
    }
#undef VCE_FUSED_ARGS
}

}  // namespace

bool ce_fused_uses_ring(int dtype, int64_t vocab) {
    // fused_dispatch: rows of more than 1024 16-byte vectors go to the ring kernel
    const int64_t nvec = dtype == VCE_BF16 ? vocab / Elem<__nv_bfloat16>::kVec : vocab / Elem<float>::kVec;
    return nvec > 1024;
}

namespace {

int row_grid(int64_t n_rows) {
    const int64_t cap = int64_t(1) << 30;
    return int(n_rows < cap ? n_rows : cap);
}

}  // namespace

vce_status launch_shift_targets(const int64_t* target, int64_t n, int64_t seq_len, int64_t ignore_idx,
                                int64_t* shifted, cudaStream_t s) {
    if (n == 0) return VCE_OK;
    const int64_t blocks = (n + 255) / 256;
    count_launch();
    shift_targets_kernel<<<int(blocks < 4096 ? blocks : 4096), 256, 0, s>>>(target, n, seq_len, ignore_idx, shifted);
    return cudaGetLastError() == cudaSuccess ? VCE_OK : VCE_ERR_CUDA;
}

vce_status launch_mean_loss(const float* loss_rows, const int64_t* target, int64_t n_rows,
                            int64_t ignore_idx, int reduce, float* loss_out, int64_t* n_valid, cudaStream_t s) {
    count_launch();
    if (!loss_rows && !loss_out && n_valid)  // the count alone
        count_valid_kernel<<<1, kCountThreads, 0, s>>>(target, n_rows, ignore_idx, n_valid);
    else
        mean_loss_kernel<false>
            <<<1, kMeanThreads, 0, s>>>(loss_rows, target, n_rows, ignore_idx, reduce, loss_out, n_valid);
    return cudaGetLastError() == cudaSuccess ? VCE_OK : VCE_ERR_CUDA;
}

vce_status launch_ce_forward(const void* logits, int dtype, int64_t n_rows, int64_t vocab,
                             int64_t row_stride, const int64_t* target, float eps,
                             int reduce_loss, int64_t ignore_idx, float* loss, float* stats,
                             int64_t* n_valid, void* ws, int* dev_status, cudaStream_t s,
                             const DeviceInfo&) {
    float* loss_rows = reduce_loss ? static_cast<float*>(ws) : loss;
    if (n_rows > 0) {
        const int grid = row_grid(n_rows);
        if (dtype == VCE_BF16)
            fwd_dispatch<__nv_bfloat16>(logits, n_rows, vocab, row_stride, target, eps, ignore_idx,
                                        loss_rows, stats, dev_status, s, grid);
        else
            fwd_dispatch<float>(logits, n_rows, vocab, row_stride, target, eps, ignore_idx,
                                loss_rows, stats, dev_status, s, grid);
        if (cudaGetLastError() != cudaSuccess) return VCE_ERR_CUDA;
    }
    if (reduce_loss || n_valid)
        return launch_mean_loss(reduce_loss ? loss_rows : nullptr, target, n_rows, ignore_idx, reduce_loss,
                                reduce_loss ? loss : nullptr, n_valid, s);
    return VCE_OK;
}

vce_status launch_ce_backward(const void* logits, int dtype, int64_t n_rows, int64_t vocab,
                              int64_t row_stride, const int64_t* target, const float* stats,
                              const int64_t* n_valid, const float* grad_output, float eps,
                              int reduce_loss, int64_t ignore_idx, void* dlogits,
                              int* dev_status, cudaStream_t s, const DeviceInfo&) {
    if (n_rows == 0) return VCE_OK;
    const int grid = row_grid(n_rows);
    if (dtype == VCE_BF16)
        bwd_dispatch<__nv_bfloat16>(logits, n_rows, vocab, row_stride, target, stats, n_valid,
                                    grad_output, eps, reduce_loss, ignore_idx, dlogits, dev_status, s, grid);
    else
        bwd_dispatch<float>(logits, n_rows, vocab, row_stride, target, stats, n_valid, grad_output,
                            eps, reduce_loss, ignore_idx, dlogits, dev_status, s, grid);
    return cudaGetLastError() == cudaSuccess ? VCE_OK : VCE_ERR_CUDA;
}

vce_status launch_ce_forward_backward(const void* logits, int dtype, int64_t n_rows, int64_t vocab,
                                      int64_t row_stride, const int64_t* target, float eps, int reduce_loss,
                                      int64_t ignore_idx, const float* grad_output, float* loss, float* stats,
                                      int64_t* n_valid, void* dlogits, void* ws, int* dev_status,
                                      cudaStream_t s, const DeviceInfo& dev, const PipeDiag& diag) {
    float* loss_rows = reduce_loss ? static_cast<float*>(ws) : loss;
    if (n_rows > 0) {
        // N_v first: the mean's upstream gradient g / N_v is needed inside the row pass
        if (reduce_loss == VCE_REDUCE_MEAN)
            if (vce_status st = launch_mean_loss(nullptr, target, n_rows, ignore_idx, reduce_loss, nullptr, n_valid, s))
                return st;
        if (dtype == VCE_BF16)
            fused_dispatch<__nv_bfloat16>(logits, n_rows, vocab, row_stride, target, eps, ignore_idx, n_valid,
                                          grad_output, reduce_loss, loss_rows, stats, dlogits, dev_status, s, dev,
                                          diag);
        else
            fused_dispatch<float>(logits, n_rows, vocab, row_stride, target, eps, ignore_idx, n_valid,
                                  grad_output, reduce_loss, loss_rows, stats, dlogits, dev_status, s, dev, diag);
        if (cudaGetLastError() != cudaSuccess) return VCE_ERR_CUDA;
        if (reduce_loss == VCE_REDUCE_MEAN) {  // N_v is in n_valid already: sum the losses alone
            count_launch();
            mean_loss_kernel<true>
                <<<1, kMeanThreads, 0, s>>>(loss_rows, target, n_rows, ignore_idx, reduce_loss, loss, n_valid);
            return cudaGetLastError() == cudaSuccess ? VCE_OK : VCE_ERR_CUDA;
        }
    }
    if (reduce_loss || n_valid)
        return launch_mean_loss(reduce_loss ? loss_rows : nullptr, target, n_rows, ignore_idx, reduce_loss,
                                reduce_loss ? loss : nullptr, n_valid, s);
    return VCE_OK;
}

}  // namespace vce
