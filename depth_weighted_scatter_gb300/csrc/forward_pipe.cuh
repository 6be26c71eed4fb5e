// forward_pipe.cuh -- the warp-specialised BEV-pooling forward (sm_103a).
//
// Computes the same thing as k_forward ("Accelerating BEV Pooling on NVIDIA
// GPUs for Physical AI Applications", sections "Eliminate redundant scatter
// traffic" and "Implement interval-owned scatter-reduce"):
//     out[bev, :] = scale * sum_{t in interval} depth[ranks_depth[t]] * feat[ranks_feat[t], :]
// with every empty cell written as zeros, each output row written once.
//
// One CTA per SM; each owns a point-balanced chunk [T0, T1) of the sorted
// map (both ends at interval starts) and a tile of cells for the zero fill.
// Its warps have three roles that run at the same time:
//
//   producers  (2 warps) stage the chunk in rounds of R points into a ring of
//              kPipeStages shared-memory stages: the three rank arrays arrive
//              by cp.async two rounds ahead; from them the producers write one
//              8-byte record per point (interval-end bit, cell, how to pick
//              the depth value out of its 32-bit word) and issue cp.async
//              copies of each point's depth word and feature row (16-byte
//              chunks, the lanes of a warp covering whole rows).  A stage's
//              "full" mbarrier completes when the records are written and
//              every copy has landed.
//   consumers  (kPipeConsWarps warps) walk each full stage exactly like the
//              compute CTAs of k_forward -- owners of LPO lanes, equal point
//              shares, a fixed-order combine of intervals cut by a share or
//              round boundary -- but read rows from shared memory, so the
//              walk never waits on L2; then they release the stage.
//   fill       (2 warps) zero the rows of the empty cells in the CTA's cell
//              tile: per sub-tile of 4096 cells, two warp-wide searches of the
//              sorted ranks_bev, a bitmap of the occupied cells, and 16-byte
//              stores of zeros to the rest.
//
// Every mbarrier wait is bounded (about half a second of %globaltimer); a
// wait that runs out counts itself in g_pipe_wait_timeouts, and from then on
// the thread stores nothing and carries on, so no warp ever waits on a warp
// that gave up and the kernel always ends.  The host reads the count with
// bevpool_forward_wait_timeouts().
#pragma once

#include <atomic>

#ifndef BEVPOOL_PIPE_STAGES
#define BEVPOOL_PIPE_STAGES 3             // shared-memory stages in the ring
#endif
#ifndef BEVPOOL_PIPE_PROD_WARPS
#define BEVPOOL_PIPE_PROD_WARPS 2         // producer warps per CTA
#endif
#ifndef BEVPOOL_PIPE_CONS_WARPS
#define BEVPOOL_PIPE_CONS_WARPS 12        // consumer warps per CTA
#endif
#ifndef BEVPOOL_PIPE_SMEM
#define BEVPOOL_PIPE_SMEM (200 * 1024)    // dynamic shared memory budget per CTA (bytes)
#endif
#ifndef BEVPOOL_PIPE_WAIT
#define BEVPOOL_PIPE_WAIT 1               // mbarrier polling: 0 try_wait, 1 test_wait, 2 try_wait with a 64 ns hint
#endif
#ifndef BEVPOOL_PIPE_BATCH
#define BEVPOOL_PIPE_BATCH 4              // points per consumer step (shared loads issued together)
#endif
#ifndef BEVPOOL_PIPE_MAX_ROUND
#define BEVPOOL_PIPE_MAX_ROUND 256        // points per round at most
#endif

namespace bevpool {

constexpr int kPipeProdWarps = BEVPOOL_PIPE_PROD_WARPS;
constexpr int kPipeFillWarps = 2;
constexpr int kPipeConsWarps = BEVPOOL_PIPE_CONS_WARPS;
constexpr int kPipeWarps = kPipeProdWarps + kPipeConsWarps + kPipeFillWarps;
constexpr int kPipeThreads = kPipeWarps * 32;
constexpr int kPipeStages = BEVPOOL_PIPE_STAGES;
constexpr int kPipeProdThreads = kPipeProdWarps * 32;
constexpr int kPipeConsThreads = kPipeConsWarps * 32;
constexpr int kPipeFillThreads = kPipeFillWarps * 32;
constexpr int kPipeFillCells = 4096;                 // cells per fill sub-tile (one bitmap)
constexpr int kBarCons = 1, kBarProd = 2, kBarFill = 3;   // named barriers (0 is __syncthreads)
constexpr long long kPipeWaitNs = 500LL * 1000 * 1000;    // bound of every mbarrier wait
static_assert(kPipeThreads <= 1024, "too many warps");

constexpr int pipe_align16(int x) { return (x + 15) / 16 * 16; }

// Shared-memory layout of one CTA (byte offsets into the dynamic buffer).
template <int DT, int C>
struct PipeLayout {
    using S = FwdShape<DT, C, kVarDefault>;
    static constexpr int ROWB = S::ROWB;
    static constexpr int CH = ROWB / 16;                  // 16-byte chunks per feature row
    static constexpr int OWNERS = kPipeConsWarps * S::OPW;
    static constexpr int SLOT_BYTES = OWNERS * C * 4;     // first partial row of every owner's share
    static constexpr int CARRY_BYTES = 2 * C * 4;         // an interval open at a round's end, by parity
    static constexpr int FIXED = SLOT_BYTES + CARRY_BYTES + OWNERS * 4 + 64 + kPipeFillCells / 8 +
                                 2 * kPipeStages * 8 + 6 * 16;
    // per point of a round: in every stage a record (8), a depth word (4) and
    // a row; in each of three rank buffers three int32 (plus a few of slack)
    static constexpr int PER_POINT = kPipeStages * (8 + 4 + ROWB) + 3 * 12;
    static constexpr int R_FIT = ((BEVPOOL_PIPE_SMEM - FIXED - 3 * 3 * 16) / PER_POINT) / 32 * 32;
    static constexpr int R = R_FIT < BEVPOOL_PIPE_MAX_ROUND ? R_FIT : BEVPOOL_PIPE_MAX_ROUND;
    static constexpr int RB = R + 4;                      // rank buffer length (ranks_bev has one extra)
    static constexpr int OFF_ROWS = 0;                                         // [stage][R][ROWB]
    static constexpr int OFF_REC = OFF_ROWS + kPipeStages * R * ROWB;          // [stage][R] uint2
    static constexpr int OFF_DW = OFF_REC + kPipeStages * R * 8;               // [stage][R] uint32
    static constexpr int OFF_RANKS = OFF_DW + kPipeStages * R * 4;             // [3][3][RB] int32
    static constexpr int OFF_SLOT = pipe_align16(OFF_RANKS + 3 * 3 * RB * 4);  // [OWNERS][C] float
    static constexpr int OFF_CARRY = OFF_SLOT + SLOT_BYTES;                    // [2][C] float
    static constexpr int OFF_STATE = OFF_CARRY + CARRY_BYTES;                  // [OWNERS] int
    static constexpr int OFF_MISC = pipe_align16(OFF_STATE + OWNERS * 4);      // 16 ints
    static constexpr int OFF_MARK = OFF_MISC + 64;                             // fill bitmap
    static constexpr int OFF_BAR = pipe_align16(OFF_MARK + kPipeFillCells / 8);   // full[S], empty[S]
    static constexpr int BYTES = OFF_BAR + 2 * kPipeStages * 8;
    static_assert(R >= 32 && R % 32 == 0, "rounds are whole warp sets of 32 points");
    static_assert(BYTES <= BEVPOOL_PIPE_SMEM, "shared-memory layout over budget");
    static_assert(ROWB % 16 == 0 && S::VB == 16, "rows are staged in 16-byte chunks, one per owner lane");
};

// Misc ints: [0, 2) carry cells by parity, [2, 4) chunk-bound search scratch,
// [4, 6) fill search results.
constexpr int kMiscCarryBev = 0, kMiscBounds = 2, kMiscFill = 4;

// ---------------------------------------------------------------- PTX helpers

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void cp_async4(uint32_t dst, const void *src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
// arrive (release): the thread's earlier shared-memory writes are visible to
// a thread whose wait observes the phase completing
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
// an arrive that happens once all of the thread's earlier cp.async copies have landed
__device__ __forceinline__ void mbar_arrive_cp_async(uint32_t bar) {
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t done;
#if BEVPOOL_PIPE_WAIT == 1
    asm volatile("{\n\t.reg .pred q;\n\tmbarrier.test_wait.parity.shared::cta.b64 q, [%1], %2;\n\t"
                 "selp.u32 %0, 1, 0, q;\n\t}"
                 : "=r"(done)
                 : "r"(bar), "r"(parity)
                 : "memory");
#elif BEVPOOL_PIPE_WAIT == 2
    asm volatile("{\n\t.reg .pred q;\n\tmbarrier.try_wait.parity.shared::cta.b64 q, [%1], %2, 64;\n\t"
                 "selp.u32 %0, 1, 0, q;\n\t}"
                 : "=r"(done)
                 : "r"(bar), "r"(parity)
                 : "memory");
#else
    asm volatile("{\n\t.reg .pred q;\n\tmbarrier.try_wait.parity.shared::cta.b64 q, [%1], %2;\n\t"
                 "selp.u32 %0, 1, 0, q;\n\t}"
                 : "=r"(done)
                 : "r"(bar), "r"(parity)
                 : "memory");
#endif
    return done != 0u;
}
__device__ __forceinline__ long long global_ns() {
    long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
__device__ __forceinline__ void named_bar_sync(int id, int n) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}

namespace {
// Waits that ran out (per compiled unit; summed by bevpool_forward_wait_timeouts).
__device__ unsigned int g_pipe_wait_timeouts;
}  // namespace

// Waits for the phase of `parity` of the mbarrier at `bar`, for at most about
// kPipeWaitNs; false (and the timeout counted) if it did not complete.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = global_ns();
    for (unsigned i = 1;; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((i & 31u) == 0u && (global_ns() - t0 > kPipeWaitNs || i >= (1u << 26))) {
            atomicAdd(&g_pipe_wait_timeouts, 1u);
            return false;
        }
    }
}

inline unsigned int pipe_wait_timeouts_here() {
    unsigned int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_pipe_wait_timeouts, sizeof(v)) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    return v;
}


// ---------------------------------------------------------------- producers

// Depth value (fp16 bits) of a point from its staged 32-bit word: `sel` is the
// byte-permute selector the producer stored in the record (fp16: the half,
// E4M3: the byte, widened exactly to fp16).
template <int DT>
__device__ __forceinline__ unsigned short pipe_depth(uint32_t word, uint32_t sel) {
    const uint32_t v = __byte_perm(word, 0u, sel & 0xffffu);
    if constexpr (DT == kDtypeF16) {
        return static_cast<unsigned short>(v);
    } else {
        return __nv_cvt_fp8_to_halfraw(static_cast<__nv_fp8_storage_t>(v & 0xffu), __NV_E4M3).x;
    }
}

// The producer warps: stage rounds [T0 + r R, ...) of the chunk into the ring.
// ptid in [0, kPipeProdThreads).
template <int DT, int C>
__device__ __forceinline__ void pipe_producer(const FwdParams &p, unsigned char *smem, int T0, int T1, int ptid) {
    using L = PipeLayout<DT, C>;
    constexpr int R = L::R;
    constexpr int K = (R + kPipeProdThreads - 1) / kPipeProdThreads;   // points per producer thread per round
    constexpr int EB = FwdShape<DT, C, kVarDefault>::EB;
    const int lane = ptid & 31, pw = ptid >> 5;
    const int nr = (T1 - T0 + R - 1) / R;
    const uint32_t sbase = smem_u32(smem);
    const uint32_t bar_full = sbase + L::OFF_BAR;
    const uint32_t bar_empty = bar_full + kPipeStages * 8;
    const unsigned char *featb = static_cast<const unsigned char *>(p.feat);
    const uintptr_t depth_addr = reinterpret_cast<uintptr_t>(p.depth);
    bool live = true;                                     // no wait of this thread has run out

    // rank buffer b: ranks_depth at [0, RB), ranks_feat at [RB, 2RB), ranks_bev at [2RB, 3RB)
    auto rank_buf = [&](int b) { return reinterpret_cast<int32_t *>(smem + L::OFF_RANKS) + b * 3 * L::RB; };
    auto issue_ranks = [&](int r) {
        if (r < nr) {
            const int t0 = T0 + r * R;
            const int cnt = min(R, T1 - t0);
            const int cntb = min(R + 1, T1 - t0);         // ranks_bev of the next point too, inside the chunk
            const uint32_t b = smem_u32(rank_buf(r % 3));
            for (int i = ptid; i < cnt; i += kPipeProdThreads) {
                cp_async4(b + 4 * i, p.ranks_depth + t0 + i);
                cp_async4(b + 4 * (L::RB + i), p.ranks_feat + t0 + i);
            }
            for (int i = ptid; i < cntb; i += kPipeProdThreads) cp_async4(b + 4 * (2 * L::RB + i), p.ranks_bev + t0 + i);
        }
        cp_async_commit();                                // one group per round, empty or not
    };

    issue_ranks(0);
    issue_ranks(1);
    for (int r = 0; r < nr; ++r) {
        const int s = r % kPipeStages;
        const int t0 = T0 + r * R;
        const int cnt = min(R, T1 - t0);
        const int cntb = min(R + 1, T1 - t0);
        // this round's ranks: groups committed after them are the previous
        // round's data and the next round's ranks (only the next ranks in round 0)
        if (r == 0) cp_async_wait<1>(); else cp_async_wait<2>();
        named_bar_sync(kBarProd, kPipeProdThreads);       // every producer's rank copies are visible
        if (r >= kPipeStages) live &= mbar_wait(bar_empty + 8 * s, ((r / kPipeStages) - 1) & 1);
        const int32_t *rb = rank_buf(r % 3);
        uint2 *rec = reinterpret_cast<uint2 *>(smem + L::OFF_REC) + s * R;
        const uint32_t dw = sbase + L::OFF_DW + 4 * s * R;
        const uint32_t rows = sbase + L::OFF_ROWS + s * R * L::ROWB;
        int rowk[K];
        bool okk[K];
#pragma unroll
        for (int k = 0; k < K; ++k) {
            const int i = ptid + k * kPipeProdThreads;
            rowk[k] = 0;
            okk[k] = false;
            if (i < cnt) {
                const int rd = rb[i], rf = rb[L::RB + i], cell = rb[2 * L::RB + i];
                const bool ok = rd >= 0 && rd < p.n_depth && rf >= 0 && rf < p.n_feat_rows;
                const bool end = i + 1 >= cntb || rb[2 * L::RB + i + 1] != cell;
                const bool nocell = !(cell >= 0 && cell < p.n_cells);
                uint32_t sel = 0x1010u;
                if (ok) {
                    // the aligned 32-bit word holding the element (it never
                    // crosses a page, so reading it is safe at either end)
                    const uintptr_t a = depth_addr + static_cast<uintptr_t>(rd) * EB;
                    cp_async4(dw + 4 * i, reinterpret_cast<const void *>(a & ~static_cast<uintptr_t>(3)));
                    const uint32_t off = static_cast<uint32_t>(a & 3);
                    sel = DT == kDtypeF16 ? (off ? 0x3232u : 0x1010u) : (0x4440u | off);
                } else {
                    asm volatile("st.shared.u32 [%0], %1;" ::"r"(dw + 4 * i), "r"(0u) : "memory");
                }
                rec[i] = make_uint2(sel | (end ? kEndBit : 0u) | (nocell ? kNoCellBit : 0u),
                                    static_cast<uint32_t>(cell));
                rowk[k] = rf;
                okk[k] = ok;
            }
        }
        // feature rows: the 32 points of a warp set are copied by the whole
        // warp, CH 16-byte chunks a row, consecutive lanes on consecutive chunks
#pragma unroll
        for (int k = 0; k < K; ++k) {
            const int base = 32 * (pw + kPipeProdWarps * k);
            if (base >= cnt) break;                        // uniform over the warp
#pragma unroll 2
            for (int j = 0; j < L::CH; ++j) {
                const int q = 32 * j + lane;
                const int pt = q / L::CH;
                const int ch = q - pt * L::CH;
                const int row = __shfl_sync(0xffffffffu, rowk[k], pt);
                const int okp = __shfl_sync(0xffffffffu, okk[k] ? 1 : 0, pt);
                const int ip = base + pt;
                if (ip < cnt) {
                    const uint32_t dst = rows + ip * L::ROWB + ch * 16;
                    if (okp)
                        cp_async16(dst, featb + static_cast<int64_t>(row) * L::ROWB + ch * 16);
                    else
                        asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(dst), "r"(0u) : "memory");
                }
            }
        }
        cp_async_commit();
        mbar_arrive_cp_async(bar_full + 8 * s);           // when this thread's copies have landed
        mbar_arrive(bar_full + 8 * s);                    // its records and zero rows are written
        issue_ranks(r + 2);
    }
    cp_async_wait_all();
    (void)live;
}

// ---------------------------------------------------------------- consumers

// The consumer warps: walk every staged round of the chunk.  ctid in
// [0, kPipeConsThreads).
template <int DT, int C, int OT>
__device__ __forceinline__ void pipe_consumer(const FwdParams &p, unsigned char *smem, int T0, int T1, int ctid) {
    using L = PipeLayout<DT, C>;
    using S = typename L::S;
    constexpr int R = L::R;
    constexpr int U = BEVPOOL_PIPE_BATCH;
    constexpr int OWNERS = L::OWNERS;
    const int lane = ctid & 31, cw = ctid >> 5;
    const int og = lane / S::LPO;                  // owner within warp
    const int ol = lane % S::LPO;                  // lane within owner
    const bool active = og < S::OPW;
    const int o = active ? cw * S::OPW + og : 0;
    float *slot = reinterpret_cast<float *>(smem + L::OFF_SLOT);     // [OWNERS][C]
    float *carry = reinterpret_cast<float *>(smem + L::OFF_CARRY);   // [2][C]
    int *state = reinterpret_cast<int *>(smem + L::OFF_STATE);
    int *carry_bev = reinterpret_cast<int *>(smem + L::OFF_MISC) + kMiscCarryBev;
    const StoreMode mode = store_mode(p.streaming != 0);
    const uint32_t bar_full = smem_u32(smem + L::OFF_BAR);
    const uint32_t bar_empty = bar_full + kPipeStages * 8;
    const int nr = (T1 - T0 + R - 1) / R;
    bool live = true;                              // no wait of this thread has run out: stores allowed
    bool round_head = true;                        // the round's first point starts an interval

    for (int r = 0; r < nr; ++r) {
        const int s = r % kPipeStages;
        const int cnt = min(R, T1 - T0 - r * R);
        const int cb = r & 1;                      // carry buffer read this round (the other is written)
        live &= mbar_wait(bar_full + 8 * s, (r / kPipeStages) & 1);
        const uint2 *rec = reinterpret_cast<const uint2 *>(smem + L::OFF_REC) + s * R;
        const uint32_t *dwp = reinterpret_cast<const uint32_t *>(smem + L::OFF_DW) + s * R;
        const unsigned char *rows = smem + L::OFF_ROWS + s * R * L::ROWB + ol * 16;
        const bool first_head = round_head;

        // owners take equal shares of the round (whole steps of U where possible)
        const int share = (cnt + OWNERS * U - 1) / (OWNERS * U) * U;
        const int beg = min(cnt, o * share);
        const int end = min(cnt, o * share + share);
        const bool next_head = (rec[cnt - 1].x & kEndBit) != 0u;
        bool head_cut = false;                     // this owner finishes an interval cut by its share end
        int head_bev = -1;
        float acc[S::EPL];                         // after the walk: the partial row of that interval
        if (active) {
            int st = kEmpty;
            if (beg < end) {
                const bool head = beg == 0 ? first_head : (rec[beg - 1].x & kEndBit) != 0u;
                bool to_slot = !head;              // the next finished segment continues a previous share
#pragma unroll
                for (int e = 0; e < S::EPL; ++e) acc[e] = 0.f;
                auto walk = [&](int v, int n, auto full_tag) {
                    constexpr bool FULL = decltype(full_tag)::value;
                    uint2 rc[U];
                    uint32_t wd[U];
                    RawVec<16> f[U];
#pragma unroll
                    for (int kk = 0; kk < U; ++kk) {
                        if (FULL || kk < n) {
                            rc[kk] = rec[v + kk];
                            wd[kk] = dwp[v + kk];
                            const uint4 q = *reinterpret_cast<const uint4 *>(rows + (v + kk) * L::ROWB);
                            f[kk].w[0] = q.x; f[kk].w[1] = q.y; f[kk].w[2] = q.z; f[kk].w[3] = q.w;
                        }
                    }
#pragma unroll
                    for (int kk = 0; kk < U; ++kk) {
                        if (FULL || kk < n) {
                            fma_vec<DT, 16>(acc, pipe_depth<DT>(wd[kk], rc[kk].x), f[kk]);
                            if (rc[kk].x & kEndBit) {          // an interval ends with this point
                                if (to_slot) {
                                    float *dst = slot + o * C + ol * S::EPL;
#pragma unroll
                                    for (int e = 0; e < S::EPL; ++e) dst[e] = acc[e];
                                    to_slot = false;
                                } else {
                                    store_interval<OT, C, S::EPL>(p, static_cast<int>(rc[kk].y), ol, acc, mode,
                                                                  live && !(rc[kk].x & kNoCellBit));
                                }
#pragma unroll
                                for (int e = 0; e < S::EPL; ++e) acc[e] = 0.f;
                            }
                        }
                    }
                };
                int v = beg;
                for (; v + U <= end; v += U) walk(v, U, std::true_type{});
                if (v < end) walk(v, end - v, std::false_type{});
                const bool cut = (rec[end - 1].x & kEndBit) == 0u;   // the share ends inside an interval
                st = head ? kHead : (to_slot && cut ? kPass : kCont);
                if (cut) {
                    if (to_slot) {                 // the whole share continues an earlier interval
                        float *dst = slot + o * C + ol * S::EPL;
#pragma unroll
                        for (int e = 0; e < S::EPL; ++e) dst[e] = acc[e];
                    } else {                       // acc keeps the interval's first part
                        head_cut = true;
                        head_bev = static_cast<int>(rec[end - 1].y);
                    }
                }
            }
            if (ol == 0) state[o] = st;
        }

        // the stage is read: release it; then combine cut intervals in owner
        // order (a fixed order, so the result is deterministic).  An interval
        // still open at the round's end goes to the carry; the first owner's
        // lanes take the carry of the previous round.
        named_bar_sync(kBarCons, kPipeConsThreads);
        if (ctid == 0) mbar_arrive(bar_empty + 8 * s);
        auto finish = [&](float *a, int o2, int bev) {
            for (; o2 < OWNERS; ++o2) {
                const int st2 = state[o2];
                if (st2 == kHead || st2 == kEmpty) break;
                const float *q = slot + o2 * C + ol * S::EPL;
#pragma unroll
                for (int e = 0; e < S::EPL; ++e) a[e] += q[e];
                if (st2 == kCont) {
                    store_interval<OT, C, S::EPL>(p, bev, ol, a, mode, live && bev >= 0 && bev < p.n_cells);
                    return;
                }
            }
            float *dst = carry + (cb ^ 1) * C + ol * S::EPL;
#pragma unroll
            for (int e = 0; e < S::EPL; ++e) dst[e] = a[e];
            if (ol == 0) carry_bev[cb ^ 1] = bev;
        };
        if (!first_head && active && o == 0) {
            float ca[S::EPL];
            const float *src = carry + cb * C + ol * S::EPL;
#pragma unroll
            for (int e = 0; e < S::EPL; ++e) ca[e] = src[e];
            finish(ca, 0, carry_bev[cb]);
        }
        if (head_cut) finish(acc, o + 1, head_bev);
        round_head = next_head;
        if (r + 1 < nr) named_bar_sync(kBarCons, kPipeConsThreads);   // the next round rewrites states and slots
    }
}

// ---------------------------------------------------------------- fill warps

// First index in [0, n) whose value is >= key in the sorted array a, by a
// 32-ary search over one warp (every lane gets the result).
__device__ __forceinline__ int warp_lower_bound(const int32_t *a, int n, int key) {
    const int lane = threadIdx.x & 31;
    int lo = 0, hi = n;
    while (hi - lo > 32) {
        const int st = (hi - lo + 31) / 32;
        const int x = lo + lane * st;
        const int c = __popc(__ballot_sync(0xffffffffu, x < hi && __ldg(a + x) < key));
        const int nlo = c > 0 ? lo + (c - 1) * st + 1 : lo;
        const int nhi = min(hi, lo + c * st);
        lo = nlo;
        hi = nhi;
    }
    const int x = lo + lane;
    return lo + __popc(__ballot_sync(0xffffffffu, x < hi && __ldg(a + x) < key));
}

// The fill warps: zero the rows of the empty cells of cells [c_begin, c_end).
// ftid in [0, kPipeFillThreads).
template <int OT, int C>
__device__ __forceinline__ void pipe_fill(const FwdParams &p, unsigned char *smem, int n_pts, int64_t c_begin,
                                          int64_t c_end, int ftid, uint32_t *mark, int *found) {
    constexpr int OUT_VECS = C * (OT == kOutF16 ? 2 : 1) / 16;     // 16-byte vectors per output row
    static_assert(OUT_VECS * 16 == C * (OT == kOutF16 ? 2 : 1), "output rows are whole 16-byte vectors");
    const int fw = ftid >> 5;
    const StoreMode mode = store_mode(p.streaming != 0);
    const uint4 z = make_uint4(0u, 0u, 0u, 0u);
    for (int64_t c0 = c_begin; c0 < c_end; c0 += kPipeFillCells) {
        const int nc = static_cast<int>(min(static_cast<int64_t>(kPipeFillCells), c_end - c0));
        for (int w = ftid; w < kPipeFillCells / 32; w += kPipeFillThreads) mark[w] = 0u;
        if (fw < 2) {                              // warp 0: first point of the sub-tile, warp 1: past it
            const int t = warp_lower_bound(p.ranks_bev, n_pts, static_cast<int>(fw == 0 ? c0 : c0 + nc));
            if ((ftid & 31) == 0) found[fw] = t;
        }
        named_bar_sync(kBarFill, kPipeFillThreads);
        const int t0 = found[0], t1 = found[1];
        for (int t = t0 + ftid; t < t1; t += kPipeFillThreads) {
            const int c = __ldg(p.ranks_bev + t) - static_cast<int>(c0);
            if (c >= 0 && c < nc) atomicOr(&mark[c >> 5], 1u << (c & 31));
        }
        named_bar_sync(kBarFill, kPipeFillThreads);
        uint4 *out = reinterpret_cast<uint4 *>(p.out) + c0 * OUT_VECS;
        const int total = nc * OUT_VECS;
        for (int v = ftid; v < total; v += kPipeFillThreads) {
            const int cell = v / OUT_VECS;
            if (!((mark[cell >> 5] >> (cell & 31)) & 1u)) store_vec(out + v, z, mode);
        }
        named_bar_sync(kBarFill, kPipeFillThreads);   // the next sub-tile clears the bitmap
    }
}

// ---------------------------------------------------------------- kernel

template <int DT, int C, int OT>
__global__ void __launch_bounds__(kPipeThreads, 1) k_forward_pipe(const FwdParams p) {
    using L = PipeLayout<DT, C>;
    grid_dep_wait();                               // the map build may still be draining (dependent launch)
    grid_dep_allow();
    extern __shared__ __align__(128) unsigned char smem[];
    const int tid = threadIdx.x, warp = tid >> 5;
    const int cidx = blockIdx.x;
    int n_int = p.n_intervals, n_pts = p.n_points;
    if (p.d_counts) {
        n_int = min(n_int, __ldg(p.d_counts + 1));
        n_pts = min(n_pts, __ldg(p.d_counts + 0));
    }
    n_pts = max(n_pts, 0);
    n_int = max(n_int, 0);
    int *misc = reinterpret_cast<int *>(smem + L::OFF_MISC);
    const uint32_t bar_full = smem_u32(smem + L::OFF_BAR);
    if (tid == 0) {
#pragma unroll
        for (int s = 0; s < kPipeStages; ++s) {
            mbar_init(bar_full + 8 * s, 2 * kPipeProdThreads);           // two arrivals per producer thread
            mbar_init(bar_full + 8 * (kPipeStages + s), 1);              // one per consumer round
        }
    }
    // the chunk: [cidx * ppc, (cidx + 1) * ppc) with both ends moved forward to
    // interval starts, so no interval is split between CTAs (uniform branch)
    int T0 = 0, T1 = 0;
    if (n_pts > 0) {
        const int ppc = static_cast<int>(p.n_compute_div.div(static_cast<uint32_t>(n_pts - 1))) + 1;
        const int64_t x0l = static_cast<int64_t>(cidx) * ppc;
        if (x0l < n_pts) {
            const int x0 = static_cast<int>(x0l);
            const int x1 = static_cast<int>(min(static_cast<int64_t>(n_pts), x0l + ppc));
            cta_next_starts(p, n_pts, n_int, x0, x1, &T0, &T1, misc + kMiscBounds);   // contains barriers
        }
    }
    __syncthreads();                               // barriers initialised
    if (warp < kPipeProdWarps) {
        if (T1 > T0) pipe_producer<DT, C>(p, smem, T0, T1, tid);
    } else if (warp < kPipeProdWarps + kPipeConsWarps) {
        if (T1 > T0) pipe_consumer<DT, C, OT>(p, smem, T0, T1, tid - kPipeProdThreads);
    } else {
        const int64_t per = (static_cast<int64_t>(p.n_cells) + p.n_compute - 1) / p.n_compute;
        const int64_t c_begin = static_cast<int64_t>(cidx) * per;
        const int64_t c_end = min(c_begin + per, static_cast<int64_t>(p.n_cells));
        pipe_fill<OT, C>(p, smem, n_pts, c_begin, c_end, tid - kPipeProdThreads - kPipeConsThreads,
                         reinterpret_cast<uint32_t *>(smem + L::OFF_MARK), misc + kMiscFill);
    }
}

// Whether the warp-specialised forward handles (DT, C): rows staged in
// 16-byte chunks (fp16 C >= 32, E4M3 C >= 64 and a multiple of 16).
template <int DT, int C>
constexpr bool pipe_supported() {
    return DT != kDtypeNVFP4 && FwdShape<DT, C, kVarDefault>::VB == 16 &&
           FwdShape<DT, C, kVarDefault>::ROWB % 16 == 0;
}

template <int DT, int C, int OT>
cudaError_t launch_forward_pipe(const ForwardArgs &a) {
    using L = PipeLayout<DT, C>;
    // the kernel's shared memory exceeds the default 48 KB: opt in once per device
    static std::atomic<unsigned long long> attr_set{0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const unsigned long long bit = 1ull << (dev & 63);
    if (!(attr_set.load(std::memory_order_acquire) & bit)) {
        e = cudaFuncSetAttribute(k_forward_pipe<DT, C, OT>, cudaFuncAttributeMaxDynamicSharedMemorySize, L::BYTES);
        if (e != cudaSuccess) return e;
        attr_set.fetch_or(bit, std::memory_order_acq_rel);
    }
    FwdParams p;
    p.depth = a.depth;
    p.feat = a.feat;
    p.feat_block = nullptr;
    p.ranks_depth = a.ranks_depth;
    p.ranks_feat = a.ranks_feat;
    p.ranks_bev = a.ranks_bev;
    p.starts = a.interval_starts;
    p.lengths = a.interval_lengths;
    p.d_counts = a.d_counts;
    p.n_points = a.n_points;
    p.n_intervals = a.n_intervals;
    p.n_cells = a.n_cells;
    p.n_feat_rows = a.n_feat_rows;
    p.n_depth = a.n_depth;
    p.scale = a.scale;
    p.streaming = a.streaming_stores;
    const int n_compute = a.sm_count > 0 ? a.sm_count : 148;   // one CTA per SM
    p.n_compute = n_compute;
    p.n_compute_div = FastDiv(static_cast<uint32_t>(n_compute));
    p.n_fill = 0;
    p.fill_cells = 0;
    p.out = static_cast<unsigned char *>(a.out);
    e = launch_dependent(k_forward_pipe<DT, C, OT>, dim3(n_compute), dim3(kPipeThreads), L::BYTES, a.stream, p);
    count_launch();
    return e;
}

}  // namespace bevpool
