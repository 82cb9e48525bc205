// Linear-form cross entropy on the tcgen05 tensor cores of sm_103a.
//
// The logits Z = X W^T are never stored (Cut Cross-Entropy card,
// "what_it_does": only the target logit and the log-sum-exp over the
// vocabulary are kept).  Every product runs through one warp-specialised GEMM
// kernel (Liger pull request "Implementation": a TMA warp feeds a multistage
// shared-memory ring, one thread issues UMMA into tensor memory, epilogue warps
// drain tensor memory), instantiated with three epilogues:
//
//   forward : Z tile -> per-(row, 256-wide vocab tile) softmax partials
//             (running max, sum of exp, sum of logits) and the target logit;
//             a small combine kernel turns the partials into lse and the loss.
//   dZ      : recomputed Z tile -> dZ = g (exp(Z - lse) - (1-eps) onehot - eps/V),
//             stored as BF16 for one vocabulary slab (backward "dZ" phase).
//   store   : plain FP32 accumulator -> BF16 (dW = dZ^T X, dX = dZ W), or an
//             FP32 running sum of dX across vocabulary slabs.
//
// Kernel shape: CTA pairs (clusters of 2) on tcgen05's cta_group::2 path.  A
// pair computes a 256 x BN output tile (BN = 256 for every product here; the
// template also builds BN = 128): each CTA stages its 128 rows of A and its
// BN/2 rows of B per 64-wide K step, the even CTA issues UMMA M=256, N=BN,
// K=16 over both CTAs' shared memory, and each CTA's tensor memory receives its
// 128 output rows.  The pair halves the B bytes every SM stages and reads,
// which buys a deeper ring (6 stages of 32 KiB) in the same shared memory.
// Persistent: one pair per two SMs; two FP32 accumulators in tensor memory so
// the epilogue of one tile overlaps the main loop of the next.  Tiles are handed
// out in order from a global ticket counter, so the tiles in progress at any
// moment are about one per pair and consecutive in the unit order; that order
// (unit_coords) groups tiles so that they share operand strips in L2.  A static
// round-robin let pairs drift apart over hundreds of tiles and multiplied the
// HBM reads at 16384 tokens (ncu: 17-21 GB for a forward of 1.2 GB of X and W).
// Warp 0: TMA producer (both CTAs).  Warp 1: tensor-memory allocation (both
// CTAs) and the MMA issuer (even CTA).  Warps 2-5: epilogue, one output row
// per thread (tensor-memory lane).
// Every mbarrier wait is bounded: past its limit (2 s) the CTA sets an abort
// flag, the other roles stop, in-flight copies and MMAs are drained, tensor
// memory is released and VCE_DEVSTATUS_TIMEOUT is reported.

#include "vce_internal.cuh"
#include "sm100_ptx.cuh"

#include <cudaTypedefs.h>
#include <math.h>
#include <mutex>
#include <type_traits>

namespace vce {
namespace {

using namespace sm100;

constexpr int BM = 256;          // output rows per CTA pair
constexpr int BM_CTA = 128;      // output rows per CTA (tensor-memory lanes)
constexpr int BK = 64;           // K elements per stage (one 128-byte swizzle row)
constexpr int kVocabTile = 256;  // forward/dZ vocabulary tile width
constexpr uint32_t kABytes = BM_CTA * BK * 2;
constexpr int kThreads = 192;
constexpr uint32_t kRingBytes = 196608;
constexpr int kUnitRing = 8;                     // work units published ahead of the slowest reader
constexpr uint32_t kUnitReaders = 10;            // odd CTA's producer, MMA issuer, 8 epilogue warps

// A pair's output tile is 256 x BN.  One MMA instruction covers N <= 256, so a
// 512-wide tile takes two per K step (pieces), each over its own 256 columns
// of B; in every piece the even CTA holds the first half of the B rows and
// the odd CTA the second.  Tiles up to 256 wide get two accumulators in
// tensor memory (the epilogue of one tile overlaps the main loop of the
// next); a 512-wide tile fills tensor memory with one, which suits products
// with a long K (dX, K = a vocabulary slab), where the epilogue is short
// beside the main loop.
template <int BN>
struct PairCfg {
    static constexpr int kMmaN = BN > 256 ? 256 : BN;        // N of one MMA instruction
    static constexpr int kPieces = BN / kMmaN;               // MMAs per 16-wide K step
    static constexpr int kPieceRows = kMmaN / 2;             // B rows this CTA stages per piece
    static constexpr uint32_t kPieceBytes = uint32_t(kPieceRows) * BK * 2;
    static constexpr uint32_t kBBytes = kPieces * kPieceBytes;  // this CTA's half of B
    static constexpr uint32_t kStageBytes = kABytes + kBBytes;
    static constexpr int kStages = (kRingBytes / kStageBytes) > 8 ? 8 : int(kRingBytes / kStageBytes);
    static constexpr int kAccs = BN > 256 ? 1 : 2;           // accumulators in tensor memory
    static constexpr uint32_t kTmemCols = kAccs * BN;
    static constexpr size_t kSmemBytes = size_t(kStages) * kStageBytes + 1024 + 512;
    static_assert(BN == 128 || BN == 256 || BN == 512, "tile width");
    static_assert(kTmemCols <= 512, "tensor memory columns");
};

struct GemmArgs {
    int tiles_m, tiles_n, k_blocks;
    int k_splits;      // the K range is cut into this many consecutive chunks (separate work units)
    int kb_per_split;  // K blocks per chunk (the last chunk may be shorter)
    int m_fastest;     // unit order: 1 = M index varies fastest, else N; the K chunk varies slowest
    int group;         // tiles of the fast index per group of the unit order (see unit_coords)
    int* counter;      // work-unit tickets, zero at launch
    int* dev_status;
    uint64_t timeout_ns;  // limit of every wait for work or data
    int hold;             // self-test only: the scheduler publishes no unit
    int64_t M, N, K;      // product extents (bounds-checking build)
};

// Work unit u -> output tile (tm, tn), K chunk ks and its K-block range [kb0, kb1).
// Units are ordered in groups of ``group`` tiles of the fast index: inside a group
// the fast index cycles over its ``group`` tiles for each value of the slow index.
// With group = all tiles of the fast index this is plain fast-index-first order.
__device__ __forceinline__ void unit_coords(const GemmArgs& a, int u, int& tm, int& tn, int& ks, int& kb0,
                                            int& kb1) {
    const int per = a.tiles_m * a.tiles_n;
    ks = u / per;
    const int t = u - ks * per;
    const int fast = a.m_fastest ? a.tiles_m : a.tiles_n;
    const int slow = a.m_fastest ? a.tiles_n : a.tiles_m;
    const int g = t / (a.group * slow);          // every group but the last has group * slow units
    const int r = t - g * (a.group * slow);
    const int f0 = g * a.group;
    const int gw = fast - f0 < a.group ? fast - f0 : a.group;
    const int f = f0 + r % gw, sl = r / gw;
    tm = a.m_fastest ? f : sl;
    tn = a.m_fastest ? sl : f;
    kb0 = ks * a.kb_per_split;
    kb1 = kb0 + a.kb_per_split;
    if (kb1 > a.k_blocks) kb1 = a.k_blocks;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 b = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&b);
}

// Store 32 consecutive floats of one row as BF16 (``left`` of them valid).
__device__ __forceinline__ void store_row32_bf16(__nv_bfloat16* dst, const float (&d)[32], int64_t left) {
    if (left >= 32) {
        uint4* q = reinterpret_cast<uint4*>(dst);
#pragma unroll
        for (int i = 0; i < 4; ++i)
            q[i] = make_uint4(pack_bf16x2(d[8 * i + 0], d[8 * i + 1]), pack_bf16x2(d[8 * i + 2], d[8 * i + 3]),
                              pack_bf16x2(d[8 * i + 4], d[8 * i + 5]), pack_bf16x2(d[8 * i + 6], d[8 * i + 7]));
    } else {
#pragma unroll
        for (int j = 0; j < 32; ++j)
            if (j < left) dst[j] = __float2bfloat16_rn(d[j]);
    }
}

// ---------------------------------------------------------------------------
// epilogues: called by every epilogue thread for its row ``gm`` of output tile
// column ``tn``; ``taddr`` is the tensor-memory address of the row's accumulator
// ---------------------------------------------------------------------------

// forward: softmax partials of one 256-wide vocabulary tile
struct FwdEpi {
    const int64_t* target;
    int64_t M;       // tokens
    int64_t V;       // vocabulary
    float2* part_ms; // [tiles_n][M] (max, sum exp(z - max))
    float* part_sum; // [tiles_n][M] sum of z (label smoothing), may be unused
    float* part_t;   // [tiles_n][M] sum of exp(z - max) z (entropy), NULL when not requested
    float* zy;       // [M] target logit
    int smooth;
    int* dev_status;

    template <int BN>
    __device__ __forceinline__ void run(int64_t gm, int tn, int ks, uint32_t taddr) const {
        static_assert(BN == kVocabTile, "partials are per 256-wide vocabulary tile");
        const bool row_ok = gm < M;
        const int64_t y = row_ok ? target[gm] : -1;
        const int64_t gn0 = int64_t(tn) * BN;
        float m = -INFINITY, negm = 0.f, s = 0.f, sum = 0.f, te = 0.f, zyv = 0.f;
        bool hit = false;
        const bool want_t = part_t != nullptr;
#pragma unroll 1
        for (int c = 0; c < BN / 32; ++c) {
            uint32_t r[32];
            tmem_ld32(taddr + c * 32, r);
            tmem_ld_wait();
            const int64_t col0 = gn0 + c * 32;
            const int64_t left = V - col0;
            float v[32];
#pragma unroll
            for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]);
            if ((uint64_t)(y - col0) < 32ull) {
#pragma unroll
                for (int j = 0; j < 32; ++j)
                    if (col0 + j == y) zyv = v[j];
                hit = true;
            }
            if (left < 32) {
#pragma unroll
                for (int j = 0; j < 32; ++j)
                    if (j >= left) v[j] = -INFINITY;
            }
            if (smooth) {
                float u = 0.f;
#pragma unroll
                for (int j = 0; j < 32; ++j) u += (j < left) ? v[j] : 0.f;
                sum += u;
            }
            float vm = v[0];
#pragma unroll
            for (int j = 1; j < 32; ++j) vm = fmaxf(vm, v[j]);
            if (vm > m) {
                const float sc = ex2f((m - vm) * kLog2e);
                s *= sc;
                te *= sc;
                m = vm;
                negm = -vm * kLog2e;
            }
            float t = 0.f, tz = 0.f;
            if (want_t) {
                // columns past V have e = 0 and an (in-range, zero-filled) raw logit of 0
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    const float e = ex2f(fmaf(v[j], kLog2e, negm));
                    t += e;
                    tz = fmaf(e, __uint_as_float(r[j]), tz);
                }
                te += tz;
            } else {
#pragma unroll
                for (int j = 0; j < 32; ++j) t += ex2f(fmaf(v[j], kLog2e, negm));
            }
            s += t;
        }
        if (row_ok && VCE_BOUNDS(tn >= 0 && int64_t(tn) * BN < V && gm >= 0, dev_status)) {
            part_ms[int64_t(tn) * M + gm] = make_float2(m, s);
            if (smooth) part_sum[int64_t(tn) * M + gm] = sum;
            if (want_t) part_t[int64_t(tn) * M + gm] = te;
            if (hit) zy[gm] = zyv;
        }
    }
};

// backward: dZ of one slab, stored BF16 [M, slab] with leading dimension ld
struct DzEpi {
    const int64_t* target;
    const float* lse;
    const float* grad;
    const int64_t* n_valid;
    int reduce;
    float eps;
    int64_t M, V, slab0, slab_cols, ld, ignore_idx;
    __nv_bfloat16* dz;
    int* dev_status;

    template <int BN>
    __device__ __forceinline__ void run(int64_t gm, int tn, int ks, uint32_t taddr) const {
        const bool row_ok = gm < M;
        bool live = false;
        int64_t y = -1;
        float g = 0.f, gp = 0.f, negl = 0.f;
        if (row_ok) {
            y = target[gm];
            const bool ign = (y == ignore_idx);
            const bool bad = !ign && (y < 0 || y >= V);
            if (bad && tn == 0 && slab0 == 0) report(dev_status, VCE_DEVSTATUS_BAD_TARGET);
            live = !ign && !bad;
            if (live) {
                g = upstream_grad(reduce, grad, n_valid, gm);
                const Exp2Offset eo = exp2_offset(lse[gm]);
                negl = eo.neg;
                gp = g * eo.fix;
            }
        }
        const float b = g * eps / float(V);
        const float c1 = g * (1.f - eps);
        const int64_t gn0 = int64_t(tn) * BN;
        __nv_bfloat16* out = dz + (row_ok ? gm : 0) * ld;
#pragma unroll 1
        for (int c = 0; c < BN / 32; ++c) {
            uint32_t r[32];
            tmem_ld32(taddr + c * 32, r);
            tmem_ld_wait();
            const int64_t col0 = gn0 + c * 32;
            const int64_t left = slab_cols - col0;
            if (!row_ok || left <= 0) continue;
            float d[32];
            if (live) {
#pragma unroll
                for (int j = 0; j < 32; ++j) d[j] = fmaf(gp, ex2f(fmaf(__uint_as_float(r[j]), kLog2e, negl)), -b);
                const int64_t yy = y - slab0 - col0;
                if ((uint64_t)yy < 32ull) {
#pragma unroll
                    for (int j = 0; j < 32; ++j) d[j] -= (j == yy) ? c1 : 0.f;
                }
            } else {
#pragma unroll
                for (int j = 0; j < 32; ++j) d[j] = 0.f;
            }
            if (VCE_BOUNDS(gm >= 0 && col0 >= 0 && col0 + (left < 32 ? left : 32) <= ld && slab0 + col0 < V,
                           dev_status))
                store_row32_bf16(out + col0, d, left);
        }
    }
};

// plain accumulator epilogue
struct StoreEpi {
    __nv_bfloat16* out;  // BF16 [M, ld_out]
    int64_t ld_out;
    float* acc;          // FP32 [k_splits][M, ld_acc] running sums across launches
    int64_t ld_acc;
    int64_t split_stride;  // elements between the FP32 buffers of consecutive K chunks
    int mode;            // 0: out = D; 1: acc = D; 2: acc += D
    int64_t M, N;
    int splits;          // K chunks, one FP32 buffer each
    int* dev_status;

    template <int BN>
    __device__ __forceinline__ void run(int64_t gm, int tn, int ks, uint32_t taddr) const {
        const bool row_ok = gm < M;
        const int64_t gn0 = int64_t(tn) * BN;
#pragma unroll 1
        for (int c = 0; c < BN / 32; ++c) {
            uint32_t r[32];
            tmem_ld32(taddr + c * 32, r);
            tmem_ld_wait();
            const int64_t col0 = gn0 + c * 32;
            const int64_t left = N - col0;
            if (!row_ok || left <= 0) continue;
            float d[32];
#pragma unroll
            for (int j = 0; j < 32; ++j) d[j] = __uint_as_float(r[j]);
            const int64_t w = left < 32 ? left : 32;
            if (mode == 0) {
                if (VCE_BOUNDS(gm >= 0 && col0 >= 0 && col0 + w <= ld_out, dev_status))
                    store_row32_bf16(out + gm * ld_out + col0, d, left);
                continue;
            }
            if (!VCE_BOUNDS(ks >= 0 && ks < splits && gm >= 0 && col0 >= 0 && col0 + w <= ld_acc, dev_status))
                continue;
            float* a = acc + int64_t(ks) * split_stride + gm * ld_acc + col0;
            if (left >= 32) {
                float4* a4 = reinterpret_cast<float4*>(a);
                if (mode == 1) {
#pragma unroll
                    for (int i = 0; i < 8; ++i) a4[i] = make_float4(d[4 * i], d[4 * i + 1], d[4 * i + 2], d[4 * i + 3]);
                } else {
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const float4 p = a4[i];
                        d[4 * i] += p.x; d[4 * i + 1] += p.y; d[4 * i + 2] += p.z; d[4 * i + 3] += p.w;
                    }
#pragma unroll
                    for (int i = 0; i < 8; ++i) a4[i] = make_float4(d[4 * i], d[4 * i + 1], d[4 * i + 2], d[4 * i + 3]);
                }
            } else {
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    if (j >= left) continue;
                    if (mode == 1) a[j] = d[j];
                    else a[j] += d[j];
                }
            }
        }
    }
};

// ---------------------------------------------------------------------------
// the GEMM: D[M, N] = A[M, K] * B[N, K]^T, BF16 in, FP32 accumulate
// A and B are K-major ([rows][K] in memory) or MN-major ([K][rows] in memory)
// ---------------------------------------------------------------------------

template <class Epi, bool kAMn, bool kBMn, int BN>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
tc_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
               const GemmArgs args, const Epi epi) {
    using C = PairCfg<BN>;
    constexpr int S = C::kStages;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + size_t(S) * C::kStageBytes);
    uint64_t* empty = full + S;
    uint64_t* tfull = empty + S;
    uint64_t* tempty = tfull + 2;
    uint64_t* drain = tempty + 2;
    uint64_t* ufull = drain + 1;             // unit ring: slot published (one arrival, the scheduler)
    uint64_t* uempty = ufull + kUnitRing;    // unit ring: slot read by every reader (even CTA's copy used)
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(uempty + kUnitRing);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    int* sched = reinterpret_cast<int*>(tmem_slot + 2);  // unit ring: the work-unit indices

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();  // 0: issues the pair's MMAs
    // (dX, dW) a GEMM launched as this one's programmatic dependent may be
    // scheduled now: its CTAs take SMs as this grid's pairs run out of work units
    // and exit
    constexpr bool kOverlaps = std::is_same<Epi, StoreEpi>::value;
    if (kOverlaps && threadIdx.x == 0) asm volatile("griddepcontrol.launch_dependents;");
    const bool leader = rank == 0;
    const int T = args.tiles_m * args.tiles_n * args.k_splits;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&tfull[b], 1);
            mbar_init(&tempty[b], 8);  // 4 epilogue warps in each CTA of the pair
        }
        mbar_init(drain, 1);
        for (int r = 0; r < kUnitRing; ++r) {
            mbar_init(&ufull[r], 1);
            mbar_init(&uempty[r], kUnitReaders);
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc_pair(tmem_slot, C::kTmemCols);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    __syncwarp();
    cluster_sync();  // barriers of both CTAs initialised before any cross-CTA signal
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    if (warp == 0) {
        if (lane == 0) {
            // ------- unit scheduler (even CTA) and TMA producer (both CTAs) -------
            // The even CTA takes work units in increasing order from a global
            // ticket counter (the next ticket is fetched while the current unit
            // loads) and publishes the pair's seq-th unit in slot seq % kUnitRing of both
            // CTAs' unit rings; a ticket >= T ends the pair's work.
            tma_prefetch_desc(&tmA);
            tma_prefetch_desc(&tmB);
            uint32_t stage = 0, phase = 0, issued = 0, issued_phase = 0;
            bool ok = true;
            int next = leader ? atomicAdd(args.counter, 1) : 0;
            // self-test of the timeout exits: no unit is published, so every
            // other role's first wait for one runs out, with nothing in flight
            if (leader && args.hold) ok = false;
            for (uint32_t seq = 0; ok; ++seq) {
                const uint32_t slot = seq % kUnitRing, upar = (seq / kUnitRing) & 1u;
                int t;
                if (leader) {
                    if (!mbar_wait<true>(&uempty[slot], upar ^ 1u, abort_flag, args.timeout_ns)) {
                        ok = false;
                        break;
                    }
                    t = next;
                    sched[slot] = t;
                    st_shared_cluster(mapa_shared(smem_u32(&sched[slot]), 1), t);
                    mbar_arrive_cluster(mapa_shared(smem_u32(&ufull[slot]), 0));
                    mbar_arrive_cluster(mapa_shared(smem_u32(&ufull[slot]), 1));
                    if (t < T) next = atomicAdd(args.counter, 1);
                } else {
                    if (!mbar_wait<true>(&ufull[slot], upar, abort_flag, args.timeout_ns)) {
                        ok = false;
                        break;
                    }
                    t = sched[slot];
                    mbar_arrive_cluster(mapa_shared(smem_u32(&uempty[slot]), 0));
                }
                if (t >= T) break;
                int tm, tn, ks, kb0, kb1;
                unit_coords(args, t, tm, tn, ks, kb0, kb1);
                const int a_row = tm * BM + int(rank) * BM_CTA;
                const int b_row = tn * BN + int(rank) * C::kPieceRows;  // first row of piece 0
                // bounds-checking build: a tensor copy starts 16-byte aligned (x, the
                // innermost coordinate, a multiple of 8 elements) inside the tile grid
                // (a box may reach past the tensor's edge: those elements read as 0);
                // a failed check skips the copy and the MMA's wait runs out
                const int64_t m_pad = int64_t(args.tiles_m) * BM, n_pad = int64_t(args.tiles_n) * BN;
                auto tma_ok = [&](int64_t x, int64_t y, int64_t x_end, int64_t y_end) {
                    return VCE_BOUNDS(x >= 0 && x % 8 == 0 && x < x_end && y >= 0 && y < y_end, args.dev_status);
                };
                for (int kb = kb0; kb < kb1; ++kb) {
                    if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag, args.timeout_ns)) {
                        ok = false;
                        break;
                    }
                    uint8_t* sa = smem + size_t(stage) * C::kStageBytes;
                    uint8_t* sb = sa + kABytes;
                    // both CTAs' copies complete on the even CTA's barrier
                    if (leader) mbar_arrive_expect_tx(&full[stage], 2 * C::kStageBytes);
                    const uint32_t fb = mapa_shared(smem_u32(&full[stage]), 0);
                    if (kAMn) {
#pragma unroll
                        for (int j = 0; j < BM_CTA / 64; ++j)
                            if (tma_ok(a_row + j * 64, kb * BK, m_pad, args.K))
                                tma_load_2d_pair(smem_u32(sa + j * 8192), &tmA, fb, a_row + j * 64, kb * BK);
                    } else if (tma_ok(kb * BK, a_row, args.K, m_pad)) {
                        tma_load_2d_pair(smem_u32(sa), &tmA, fb, kb * BK, a_row);
                    }
#pragma unroll
                    for (int pc = 0; pc < C::kPieces; ++pc) {
                        const int row = b_row + pc * C::kMmaN;
                        uint8_t* dst = sb + pc * C::kPieceBytes;
                        if (kBMn) {
#pragma unroll
                            for (int j = 0; j < C::kPieceRows / 64; ++j)
                                if (tma_ok(row + j * 64, kb * BK, n_pad, args.K))
                                    tma_load_2d_pair(smem_u32(dst + j * 8192), &tmB, fb, row + j * 64, kb * BK);
                        } else if (tma_ok(kb * BK, row, args.K, n_pad)) {
                            tma_load_2d_pair(smem_u32(dst), &tmB, fb, kb * BK, row);
                        }
                    }
                    issued |= 1u << stage;
                    issued_phase = (issued_phase & ~(1u << stage)) | (phase << stage);
                    if (++stage == uint32_t(S)) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            if (!ok && leader) {
                // let copies already in flight land before shared memory is released
                volatile int no_abort = 0;
                for (int s = 0; s < S; ++s)
                    if ((issued >> s) & 1u)
                        mbar_wait(&full[s], (issued_phase >> s) & 1u, &no_abort, kDrainTimeoutNs);
            }
        }
    } else if (warp == 1) {
        if (lane == 0 && leader) {
            // ---------------- MMA issuer (even CTA) ----------------
            constexpr uint32_t kIdesc = idesc_bf16_f32(BM, C::kMmaN, kAMn, kBMn);
            uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
            bool ok = true;
            for (uint32_t seq = 0; ok; ++seq) {
                const uint32_t slot = seq % kUnitRing, upar = (seq / kUnitRing) & 1u;
                if (!mbar_wait<true>(&ufull[slot], upar, abort_flag, args.timeout_ns)) break;
                const int t = sched[slot];
                mbar_arrive_cluster(mapa_shared(smem_u32(&uempty[slot]), 0));
                if (t >= T) break;
                int tm, tn, ks, kb0, kb1;
                unit_coords(args, t, tm, tn, ks, kb0, kb1);
                if (!mbar_wait(&tempty[acc], acc_phase ^ 1u, abort_flag, args.timeout_ns)) break;
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + acc * BN;
                for (int kb = kb0; kb < kb1; ++kb) {
                    if (!mbar_wait(&full[stage], phase, abort_flag, args.timeout_ns)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sa = smem_u32(smem + size_t(stage) * C::kStageBytes);
                    const uint32_t sb = sa + kABytes;
#pragma unroll
                    for (int kk = 0; kk < BK / 16; ++kk) {
                        const uint64_t ad = kAMn ? smem_desc_sw128(sa + kk * 2048, 8192, 1024)
                                                 : smem_desc_sw128(sa + kk * 32, 16, 1024);
#pragma unroll
                        for (int pc = 0; pc < C::kPieces; ++pc) {
                            const uint32_t sbp = sb + pc * C::kPieceBytes;
                            const uint64_t bd = kBMn ? smem_desc_sw128(sbp + kk * 2048, 8192, 1024)
                                                     : smem_desc_sw128(sbp + kk * 32, 16, 1024);
                            umma_bf16_pair(d_tmem + pc * C::kMmaN, ad, bd, kIdesc, (kb > kb0 || kk > 0) ? 1u : 0u);
                        }
                    }
                    umma_commit_pair(&empty[stage], 0x3);  // frees the stage in both CTAs
                    if (++stage == uint32_t(S)) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                umma_commit_pair(&tfull[acc], 0x3);
                if (++acc == uint32_t(C::kAccs)) {
                    acc = 0;
                    acc_phase ^= 1u;
                }
            }
            // every MMA issued so far completes before tensor memory is released
            umma_commit_pair(drain, 0x1);
            volatile int no_abort = 0;
            mbar_wait(drain, 0, &no_abort, kDrainTimeoutNs);
        }
    } else {
        // ---------------- epilogue (warps 2..5 of both CTAs) ----------------
        const int q = warp & 3;  // tensor-memory lane quadrant this warp may access
        const uint32_t tempty_leader[2] = {mapa_shared(smem_u32(&tempty[0]), 0), mapa_shared(smem_u32(&tempty[1]), 0)};
        uint32_t acc = 0, acc_phase = 0;
        for (uint32_t seq = 0;; ++seq) {
            const uint32_t slot = seq % kUnitRing, upar = (seq / kUnitRing) & 1u;
            bool ok = mbar_wait<true>(&ufull[slot], upar, abort_flag, args.timeout_ns);
            if (!__all_sync(0xffffffffu, ok)) break;
            const int t = sched[slot];
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(mapa_shared(smem_u32(&uempty[slot]), 0));
            if (t >= T) break;
            ok = mbar_wait(&tfull[acc], acc_phase, abort_flag, args.timeout_ns);
            if (!__all_sync(0xffffffffu, ok)) break;
            tc_fence_after();
            int tm, tn, ks, kb0, kb1;
            unit_coords(args, t, tm, tn, ks, kb0, kb1);
            const uint32_t taddr = tmem_base + (uint32_t(q * 32) << 16) + acc * BN;
            epi.template run<BN>(int64_t(tm) * BM + int64_t(rank) * BM_CTA + q * 32 + lane, tn, ks, taddr);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(tempty_leader[acc]);
            if (++acc == uint32_t(C::kAccs)) {
                acc = 0;
                acc_phase ^= 1u;
            }
        }
    }

    __syncthreads();
    if (threadIdx.x == 0 && *abort_flag) report(args.dev_status, VCE_DEVSTATUS_TIMEOUT);
    tc_fence_before();
    __syncwarp();
    cluster_sync();  // the pair is done: no more MMAs, copies or remote arrivals
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair(tmem_base, C::kTmemCols);
    }
    // A GEMM launched to overlap the tail of the previous one (programmatic
    // dependent launch) completes only after that one: later work on the stream
    // may then rely on both.  Without such a prerequisite this returns at once.
    if (kOverlaps && threadIdx.x == 0) asm volatile("griddepcontrol.wait;" ::: "memory");
}

// ---------------------------------------------------------------------------
// forward combine: partials of every vocabulary tile -> lse, loss
// ---------------------------------------------------------------------------

constexpr int kCombRows = 32;   // consecutive rows per CTA (coalesced partial reads)
constexpr int kCombSplit = 8;   // partial-index splits per row, merged in a fixed order

// merge (m2, s2, t2) into (m, s, t): s = sum exp(z - m), t = sum exp(z - m) z
__device__ __forceinline__ void lse_merge(float& m, float& s, float& t, float m2, float s2, float t2) {
    const float mn = fmaxf(m, m2);
    if (mn == -INFINITY) return;
    const float a = ex2f((m - mn) * kLog2e), b = ex2f((m2 - mn) * kLog2e);
    s = s * a + s2 * b;
    t = t * a + t2 * b;
    m = mn;
}

__global__ void __launch_bounds__(kCombRows * kCombSplit)
lce_combine_kernel(const float2* __restrict__ part_ms, const float* __restrict__ part_sum,
                   const float* __restrict__ part_t, const float* __restrict__ zy,
                   const int64_t* __restrict__ target, int64_t n, int64_t v, int nb, float eps,
                   int64_t ignore_idx, float* __restrict__ lse_out, float* __restrict__ loss_out,
                   float* __restrict__ entropy_out, int* dev_status) {
    __shared__ float sm_m[kCombSplit][kCombRows], sm_s[kCombSplit][kCombRows], sm_u[kCombSplit][kCombRows],
        sm_t[kCombSplit][kCombRows];
    const int lr = threadIdx.x % kCombRows, sp = threadIdx.x / kCombRows;
    const int64_t row = int64_t(blockIdx.x) * kCombRows + lr;
    const bool want_t = entropy_out != nullptr;
    float m = -INFINITY, s = 0.f, u = 0.f, t = 0.f;
    if (row < n) {
        // eight partials per batch with every load issued before the merges (the
        // merge order is unchanged): a load per dependent merge left each load's
        // latency exposed, 35.5 against 16.0 us at 4096 rows x 512 tiles
        constexpr int U = 8;
        int b = sp;
        for (; b + (U - 1) * kCombSplit < nb; b += U * kCombSplit) {
            float2 p[U];
            float pt[U], pu[U];
#pragma unroll
            for (int k = 0; k < U; ++k) {
                const int64_t idx = int64_t(b + k * kCombSplit) * n + row;
                p[k] = part_ms[idx];
                pt[k] = want_t ? part_t[idx] : 0.f;
                pu[k] = eps != 0.f ? part_sum[idx] : 0.f;
            }
#pragma unroll
            for (int k = 0; k < U; ++k) {
                lse_merge(m, s, t, p[k].x, p[k].y, pt[k]);
                if (eps != 0.f) u += pu[k];
            }
        }
        for (; b < nb; b += kCombSplit) {
            const float2 p = part_ms[int64_t(b) * n + row];
            lse_merge(m, s, t, p.x, p.y, want_t ? part_t[int64_t(b) * n + row] : 0.f);
            if (eps != 0.f) u += part_sum[int64_t(b) * n + row];
        }
    }
    sm_m[sp][lr] = m;
    sm_s[sp][lr] = s;
    sm_u[sp][lr] = u;
    sm_t[sp][lr] = t;
    __syncthreads();
    if (sp != 0 || row >= n) return;
    for (int k = 1; k < kCombSplit; ++k) {
        lse_merge(m, s, t, sm_m[k][lr], sm_s[k][lr], sm_t[k][lr]);
        u += sm_u[k][lr];
    }
    const float lse = m + logf(s);
    lse_out[row] = lse;
    if (want_t) entropy_out[row] = lse - t / s;  // H = lse - sum_v p_v z_v
    const int64_t y = target[row];
    float loss;
    if (y == ignore_idx) {
        loss = 0.f;
    } else if (y < 0 || y >= v) {
        loss = __int_as_float(0x7fc00000);
        report(dev_status, VCE_DEVSTATUS_BAD_TARGET);
    } else {
        loss = lse - zy[row];
        if (eps != 0.f) loss = (1.f - eps) * loss + eps * (lse - u / float(v));
    }
    loss_out[row] = loss;
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// 2-D BF16 tensor map: ``inner`` contiguous elements per row, ``outer`` rows of
// ``row_bytes`` bytes; box of box_inner x box_outer elements, 128-byte swizzle,
// zero fill out of bounds.
bool make_map(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer, uint64_t row_bytes,
              uint32_t box_inner, uint32_t box_outer) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {row_bytes};
    cuuint32_t box[2] = {box_inner, box_outer};
    cuuint32_t es[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// K-major operand: rows of K elements; box = 64 K x ``rows_box`` rows
bool map_kmajor(CUtensorMap* m, const void* base, int64_t k, int64_t rows, int64_t ld, uint32_t rows_box) {
    return make_map(m, base, uint64_t(k), uint64_t(rows), uint64_t(ld) * 2, BK, rows_box);
}

// MN-major operand: rows of MN elements, one row per K index; box = 64 x 64
bool map_mnmajor(CUtensorMap* m, const void* base, int64_t mn, int64_t k, int64_t ld) {
    return make_map(m, base, uint64_t(mn), uint64_t(k), uint64_t(ld) * 2, 64, BK);
}

// Zeroes ``count`` work-unit counters (a kernel rather than a memset, so that
// the reset is ordered on the compute stream like the GEMMs and never waits
// behind copies that another stream has queued on a copy engine).
__global__ void reset_counter_kernel(int* counter, int count) {
    for (int i = 0; i < count; ++i) counter[i] = 0;
}

// How launch_gemm orders a GEMM after the work before it on the stream.
enum class After {
    kReset,    // zero the counter first (one small kernel), then a plain launch
    kPlain,    // the counter was zeroed earlier; plain launch
    kOverlap,  // the counter was zeroed earlier; programmatic dependent launch:
               // the GEMM starts on SMs the previous GEMM's pairs leave, so it
               // must not read that GEMM's results (it reads none of them)
};

// Tiles of the fast index per group of the unit order.  The group's strips of the
// fast-index operand (A when M is fast, B when N is: 256 rows x the unit's K range)
// are read by every unit of the group, and each strip of the other operand by
// ``group`` consecutive units, so the fast operand is read from HBM once and the
// other once per group.  The group is as wide as a third of L2 holds, and never
// narrower than about sqrt(CTA pairs) tiles: when strips are too long for L2
// (K = a vocabulary slab), the pairs working at one time then still cover a
// near-square block of output tiles and share their strips while they stream.
// ``aspect`` is the fast index's tile extent over the slow index's (BM / BN when
// M is fast): a block of ``pairs`` tiles g fast x (pairs / g) slow covers the
// fewest operand rows at g = sqrt(pairs / aspect).
int raster_group(int tiles_fast, int64_t strip_bytes, double aspect, const DeviceInfo& dev) {
    const int pairs = dev.num_sms / 2;
    int g_win = 1;
    while (double(g_win) * g_win * aspect < pairs) ++g_win;
    const int64_t budget = int64_t(dev.l2_bytes / 3);
    const int64_t g_l2 = strip_bytes > 0 ? budget / strip_bytes : tiles_fast;
    int64_t g = g_l2 > g_win ? g_l2 : g_win;
    if (g >= tiles_fast) return tiles_fast < 1 ? 1 : tiles_fast;
    const int64_t groups = (tiles_fast + g - 1) / g;  // equal groups, as few as that width allows
    return int((tiles_fast + groups - 1) / groups);
}

template <class Epi, bool kAMn, bool kBMn, int BN>
vce_status launch_gemm(const CUtensorMap& a, const CUtensorMap& b, int64_t M, int64_t N, int64_t K, int m_fastest,
                       int k_splits, const Epi& epi, int* counter, int* dev_status, cudaStream_t s,
                       const DeviceInfo& dev, const PipeDiag& diag = PipeDiag(), After after = After::kReset) {
    using C = PairCfg<BN>;
    auto kern = tc_gemm_kernel<Epi, kAMn, kBMn, BN>;
    // the shared-memory limit is a per-device attribute of the kernel: raise it
    // once on every device this instantiation runs on
    static std::mutex mu;
    static bool raised[64] = {};
    if (dev.ordinal < 0 || dev.ordinal >= 64) return VCE_ERR_CUDA;
    {
        std::lock_guard<std::mutex> lock(mu);
        if (!raised[dev.ordinal]) {
            if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(C::kSmemBytes)) !=
                cudaSuccess)
                return VCE_ERR_CUDA;
            raised[dev.ordinal] = true;
        }
    }
    GemmArgs args;
    args.tiles_m = int((M + BM - 1) / BM);
    args.tiles_n = int((N + BN - 1) / BN);
    args.k_blocks = int((K + BK - 1) / BK);
    if (k_splits < 1) k_splits = 1;
    if (k_splits > args.k_blocks) k_splits = args.k_blocks;
    args.kb_per_split = (args.k_blocks + k_splits - 1) / k_splits;
    args.k_splits = (args.k_blocks + args.kb_per_split - 1) / args.kb_per_split;  // every chunk non-empty
    args.m_fastest = m_fastest;
    {
        const int64_t strip = int64_t(m_fastest ? BM : BN) * args.kb_per_split * BK * 2;
        const double aspect = m_fastest ? double(BM) / BN : double(BN) / BM;
        args.group = raster_group(m_fastest ? args.tiles_m : args.tiles_n, strip, aspect, dev);
    }
    args.counter = counter;
    args.dev_status = dev_status;
    args.timeout_ns = diag.timeout_ns;
    args.hold = diag.hold;
    args.M = M;
    args.N = N;
    args.K = K;
    const int64_t units = int64_t(args.tiles_m) * args.tiles_n * args.k_splits;
    if (units <= 0 || args.k_blocks <= 0) return VCE_OK;
    const int64_t pairs = dev.num_sms / 2;
    const int grid = 2 * int(units < pairs ? units : pairs);
    if (after == After::kReset) {
        count_launch();
        reset_counter_kernel<<<1, 1, 0, s>>>(counter, 1);
    }
    count_launch();
    if (after == After::kOverlap) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(grid);
        cfg.blockDim = dim3(kThreads);
        cfg.dynamicSmemBytes = C::kSmemBytes;
        cfg.stream = s;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        if (cudaLaunchKernelEx(&cfg, kern, a, b, args, epi) == cudaSuccess) return VCE_OK;
        (void)cudaGetLastError();  // not accepted here: the plain launch below
    }
    kern<<<grid, kThreads, C::kSmemBytes, s>>>(a, b, args, epi);
    return cudaGetLastError() == cudaSuccess ? VCE_OK : VCE_ERR_CUDA;
}

// Number of K chunks for the dX GEMM (K = vocabulary slab): the smallest count
// in 1..4 whose work units fill the CTA pairs' last round best.
int dx_k_splits(int64_t n, int64_t h, int bn, int num_sms) {
    const int64_t tiles = ((n + BM - 1) / BM) * ((h + bn - 1) / bn);
    const int64_t pairs = num_sms / 2;
    int best = 1;
    double best_eff = 0.0;
    for (int s = 1; s <= 4; ++s) {
        const int64_t units = tiles * s;
        const int64_t rounds = (units + pairs - 1) / pairs;
        const double e = double(units) / double(rounds * pairs);
        if (e > best_eff + 0.02) {
            best_eff = e;
            best = s;
        }
    }
    return best;
}

// Tile width and K chunks of the dX GEMM (dX = dZ W: M = tokens, N = hidden,
// K = a vocabulary slab of ``slab`` ids).  With 512-wide tiles each 256-token
// strip of dZ is read once per 512 hidden columns instead of once per 256: less
// DRAM and L2 traffic, which under the power cap buys clock (same-box A/B runs:
// 1-4% faster steps at 2048-4096 tokens even where its fewer units fill the
// pairs' rounds worse).  Its single accumulator leaves the epilogue (an FP32
// partial of 256 x 512) outside the main loop, which costs little only when
// each work unit runs over a long K range, so the wide tile takes the chunk
// count that fills the rounds best among those that keep chunks of at least
// 16384 vocabulary ids (hidden sizes of at least two tiles).  Otherwise the
// 256-wide tile, with the chunk count of dx_k_splits.
struct DxPlan {
    int tile_n, splits;
};

DxPlan dx_plan(int64_t n, int64_t h, int64_t slab, int num_sms) {
    if (h >= 1024) {
        const int64_t tiles = ((n + BM - 1) / BM) * ((h + 511) / 512);
        const int64_t pairs = num_sms / 2;
        int best = 0;
        double best_eff = 0.0;
        for (int s = 1; s <= 4 && slab / s >= 16384; ++s) {
            const int64_t units = tiles * s;
            const int64_t rounds = (units + pairs - 1) / pairs;
            const double e = double(units) / double(rounds * pairs);
            if (e > best_eff + 0.02) {
                best_eff = e;
                best = s;
            }
        }
        if (best > 0) return {512, best};
    }
    return {256, dx_k_splits(n, h, 256, num_sms)};
}

// Tile width of the dW GEMM (dW_slab = dZ^T X: M = slab ids, N = hidden, K =
// tokens).  Each work unit streams a strip of the slab's dZ and one of X over all
// tokens; with 512-wide tiles the CTA pairs working at one time cover half as
// many hidden tiles, so each round reads fewer X strips, and the tile's single
// accumulator leaves its epilogue outside the main loop, which K ranges of
// kDwWideTokens tokens or more amortise.
constexpr int64_t kDwWideTokens = 8192;

int dw_tile(int64_t n, int64_t h) { return n >= kDwWideTokens && h >= 1024 ? 512 : 256; }

// dX = sum of the FP32 partials of every K chunk, rounded to BF16 (fixed order).
__global__ void dx_finalize_kernel(const float* __restrict__ acc, int splits, int64_t split_stride,
                                   int64_t count4, __nv_bfloat16* __restrict__ dx) {
    for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < count4; i += int64_t(gridDim.x) * blockDim.x) {
        float4 v = reinterpret_cast<const float4*>(acc)[i];
        for (int k = 1; k < splits; ++k) {
            const float4 w = reinterpret_cast<const float4*>(acc + k * split_stride)[i];
            v.x += w.x; v.y += w.y; v.z += w.z; v.w += w.w;
        }
        reinterpret_cast<uint2*>(dx)[i] = make_uint2(pack_bf16x2(v.x, v.y), pack_bf16x2(v.z, v.w));
    }
}

struct FwdWs {
    float2* part_ms;
    float* part_sum;
    float* part_t;
    float* zy;
    float* loss_rows;
    int* counter;
    size_t bytes;
};

FwdWs carve_forward(void* ws, int64_t n, int64_t v, int reduce_loss) {
    const int64_t nb = (v + kVocabTile - 1) / kVocabTile;
    FwdWs w{};
    size_t off = 0;
    uint8_t* base = static_cast<uint8_t*>(ws);
    w.part_ms = reinterpret_cast<float2*>(base + off);
    off += align256(size_t(nb) * size_t(n) * 8);
    w.part_sum = reinterpret_cast<float*>(base + off);
    off += align256(size_t(nb) * size_t(n) * 4);
    w.part_t = reinterpret_cast<float*>(base + off);
    off += align256(size_t(nb) * size_t(n) * 4);
    w.zy = reinterpret_cast<float*>(base + off);
    off += align256(size_t(n) * 4);
    w.loss_rows = reduce_loss ? reinterpret_cast<float*>(base + off) : nullptr;
    if (reduce_loss) off += align256(size_t(n) * 4);
    w.counter = reinterpret_cast<int*>(base + off);
    off += 256;
    w.bytes = off;
    return w;
}

int64_t slab_ld(int64_t slab) { return (slab + 7) / 8 * 8; }

// Backward workspace: the BF16 dZ slab, then (unless one slab and one K chunk
// let dX be written directly) the FP32 dX partial sums of every K chunk, then
// 256 bytes for the GEMMs' work-unit counters (the forward's and dZ's in the first int, dX's and dW's in the first two).
struct BwdPlan {
    int64_t ld;      // dZ slab leading dimension
    int splits;      // K chunks of the dX GEMM
    int tile_n;      // width of the dX GEMM's pair tile (every slab)
    bool direct;     // dX written as BF16 by the GEMM itself
    size_t dz_bytes, acc_bytes;
};

BwdPlan plan_backward(int64_t n, int64_t h, int64_t v, int64_t slab, int num_sms) {
    BwdPlan p;
    p.ld = slab_ld(slab);
    // the chunk count the dX launch of the first (widest) slab really uses:
    // at most one chunk per 64-wide K block, every chunk non-empty
    const int64_t kb = ((slab < v ? slab : v) + BK - 1) / BK;
    const DxPlan dp = dx_plan(n, h, slab < v ? slab : v, num_sms);
    p.tile_n = dp.tile_n;
    int splits = dp.splits;
    if (splits > kb) splits = int(kb);
    const int64_t per = (kb + splits - 1) / splits;
    p.splits = int((kb + per - 1) / per);
    p.direct = slab >= v && p.splits == 1;
    p.dz_bytes = align256(size_t(n) * size_t(p.ld) * 2);
    p.acc_bytes = p.direct ? 0 : align256(size_t(p.splits) * size_t(n) * size_t(h) * 4);
    return p;
}

int planning_sms() {
    DeviceInfo d;
    return current_device(d) == VCE_OK ? d.num_sms : 152;
}

}  // namespace

size_t lce_forward_ws_bytes(int64_t n, int64_t v, int reduce_loss) {
    return carve_forward(nullptr, n, v, reduce_loss).bytes;
}

size_t lce_backward_ws_bytes(int64_t n, int64_t h, int64_t v, int64_t slab) {
    const BwdPlan p = plan_backward(n, h, v, slab, planning_sms());
    return p.dz_bytes + p.acc_bytes + 256;
}

int64_t lce_slab_for_ws(int64_t n, int64_t h, int64_t v, size_t ws_bytes) {
    if (ws_bytes >= lce_backward_ws_bytes(n, h, v, v)) return v;
    int64_t cap = v / 256 * 256;
    if (cap < 256) cap = 256;
    while (cap >= 256 && lce_backward_ws_bytes(n, h, v, cap) > ws_bytes) {
        const int64_t guess = int64_t(ws_bytes / (size_t(n) * 2)) / 256 * 256;
        cap = (guess < cap - 256) ? guess : cap - 256;
    }
    if (cap < 256) return 0;
    return cap < v ? cap : v;
}

vce_status launch_lce_forward(const void* X, const void* W, int64_t n, int64_t h, int64_t v,
                              const int64_t* target, float eps, int reduce_loss, int64_t ignore_idx,
                              float* loss, float* lse, float* entropy, int64_t* n_valid, void* ws,
                              int* dev_status, cudaStream_t s, const DeviceInfo& dev, const PipeDiag& diag) {
    if (n == 0) {
        if (reduce_loss || n_valid)
            return launch_mean_loss(nullptr, target, 0, ignore_idx, reduce_loss, reduce_loss ? loss : nullptr,
                                    n_valid, s);
        return VCE_OK;
    }
    const FwdWs w = carve_forward(ws, n, v, reduce_loss);
    CUtensorMap tx, tw;
    if (!map_kmajor(&tx, X, h, n, h, BM_CTA) || !map_kmajor(&tw, W, h, v, h, kVocabTile / 2)) return VCE_ERR_CUDA;
    FwdEpi epi{target, n, v, w.part_ms, w.part_sum, entropy ? w.part_t : nullptr, w.zy, eps != 0.f ? 1 : 0,
               dev_status};
    if (vce_status st =
            launch_gemm<FwdEpi, false, false, kVocabTile>(tx, tw, n, v, h, 1, 1, epi, w.counter, dev_status, s, dev,
                                                          diag))
        return st;
    const int nb = int((v + kVocabTile - 1) / kVocabTile);
    float* loss_rows = reduce_loss ? w.loss_rows : loss;
    count_launch();
    lce_combine_kernel<<<int((n + kCombRows - 1) / kCombRows), kCombRows * kCombSplit, 0, s>>>(
        w.part_ms, w.part_sum, w.part_t, w.zy, target, n, v, nb, eps, ignore_idx, lse, loss_rows, entropy,
        dev_status);
    if (cudaGetLastError() != cudaSuccess) return VCE_ERR_CUDA;
    if (reduce_loss || n_valid)
        return launch_mean_loss(reduce_loss ? loss_rows : nullptr, target, n, ignore_idx, reduce_loss,
                                reduce_loss ? loss : nullptr, n_valid, s);
    return VCE_OK;
}

vce_status launch_lce_backward(const void* X, const void* W, int64_t n, int64_t h, int64_t v,
                               const int64_t* target, const float* lse, const int64_t* n_valid,
                               const float* grad_output, float eps, int reduce_loss, int64_t ignore_idx,
                               void* dX, void* dW, void* ws, int64_t slab, int* dev_status, cudaStream_t s,
                               const DeviceInfo& dev) {
    if (n == 0) {
        return cudaMemsetAsync(dW, 0, size_t(v) * size_t(h) * 2, s) == cudaSuccess ? VCE_OK : VCE_ERR_CUDA;
    }
    const BwdPlan plan = plan_backward(n, h, v, slab, dev.num_sms);
    const int64_t ld = plan.ld;
    auto* dz = static_cast<__nv_bfloat16*>(ws);
    float* acc = plan.direct ? nullptr : reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + plan.dz_bytes);
    int* counter = reinterpret_cast<int*>(static_cast<uint8_t*>(ws) + plan.dz_bytes + plan.acc_bytes);
    const int64_t split_stride = n * h;
    const auto* Wb = static_cast<const __nv_bfloat16*>(W);
    auto* dWb = static_cast<__nv_bfloat16*>(dW);
    auto* dXb = static_cast<__nv_bfloat16*>(dX);
    CUtensorMap tx_k, tx_mn;
    if (!map_kmajor(&tx_k, X, h, n, h, BM_CTA) || !map_mnmajor(&tx_mn, X, h, n, h)) return VCE_ERR_CUDA;
    for (int64_t v0 = 0; v0 < v; v0 += slab) {
        const int64_t vs = (v - v0) < slab ? (v - v0) : slab;
        // dZ = epilogue(X W_slab^T): M = n, N = vs, K = h
        CUtensorMap tws_k, tdz_k, tdz_mn, tws_mn;
        if (!map_kmajor(&tws_k, Wb + v0 * h, h, vs, h, kVocabTile / 2) || !map_kmajor(&tdz_k, dz, vs, n, ld, BM_CTA) ||
            !map_mnmajor(&tdz_mn, dz, vs, n, ld) || !map_mnmajor(&tws_mn, Wb + v0 * h, h, vs, h))
            return VCE_ERR_CUDA;
        DzEpi de{target, lse, grad_output, n_valid, reduce_loss, eps, n, v, v0, vs, ld, ignore_idx, dz, dev_status};
        if (vce_status st =
                launch_gemm<DzEpi, false, false, kVocabTile>(tx_k, tws_k, n, vs, h, 1, 1, de, counter, dev_status, s,
                                                             dev))
            return st;
        // dX and dW both read only the dZ slab.  dX goes first, on counter[0]: its
        // few long work units leave pairs idle in its last round, and dW, on
        // counter[1], is launched to overlap that tail (its CTAs take the SMs the
        // dX pairs leave).  Each GEMM grid completes only after its prerequisite,
        // so the next slab's dZ and the dX finalize follow both.
        count_launch();
        reset_counter_kernel<<<1, 1, 0, s>>>(counter, 2);
        // dX (+)= dZ W_slab: M = n, N = h, K = vs (W_slab read MN-major), K cut into plan.splits chunks
        StoreEpi xe{dXb, h, acc, h, split_stride, plan.direct ? 0 : (v0 == 0 ? 1 : 2), n, h, plan.splits, dev_status};
        const vce_status sx =
            plan.tile_n == 512
                ? launch_gemm<StoreEpi, false, true, 512>(tdz_k, tws_mn, n, h, vs, 1, plan.splits, xe, counter,
                                                          dev_status, s, dev, PipeDiag(), After::kPlain)
                : launch_gemm<StoreEpi, false, true, 256>(tdz_k, tws_mn, n, h, vs, 1, plan.splits, xe, counter,
                                                          dev_status, s, dev, PipeDiag(), After::kPlain);
        if (sx != VCE_OK) return sx;
        // dW_slab = dZ^T X: M = vs, N = h, K = n (both operands MN-major)
        StoreEpi we{dWb + v0 * h, h, nullptr, 0, 0, 0, vs, h, 1, dev_status};
        const vce_status sw =
            dw_tile(n, h) == 512
                ? launch_gemm<StoreEpi, true, true, 512>(tdz_mn, tx_mn, vs, h, n, 0, 1, we, counter + 1, dev_status, s,
                                                         dev, PipeDiag(), After::kOverlap)
                : launch_gemm<StoreEpi, true, true, 256>(tdz_mn, tx_mn, vs, h, n, 0, 1, we, counter + 1, dev_status, s,
                                                         dev, PipeDiag(), After::kOverlap);
        if (sw != VCE_OK) return sw;
    }
    if (!plan.direct) {
        const int64_t count4 = n * h / 4;  // h is a multiple of 8
        const int blocks = int((count4 + 255) / 256 < 4096 ? (count4 + 255) / 256 : 4096);
        count_launch();
        dx_finalize_kernel<<<blocks, 256, 0, s>>>(acc, plan.splits, split_stride, count4, dXb);
        if (cudaGetLastError() != cudaSuccess) return VCE_ERR_CUDA;
    }
    return VCE_OK;
}

}  // namespace vce
