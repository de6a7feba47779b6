// ep_layout kernels: expert histogram, padded exclusive scan, stable slots.
//
// The layout step that DeepEP V2's dispatch performs internally ("infers the
// layout from topk_idx", SGLang PR "moe: add DeepEP V2 ElasticBuffer support
// to MoE token dispatcher", section "Motivation"), for the contiguous
// (prefill) and masked (decode) layouts of SGLang PR "[Feature] Add DeepEPv2
// (ElasticBuffer) MoE A2A backend", section "Supported scope".
//
// Design (deterministic, no global atomics on slot order; latency-bound, so
// the goal is short dependency chains and many warps):
//   * the T*K entries are cut into tiles; warp w of a tile's CTA owns a
//     contiguous chunk of at most 256 entries, lane l holds entries
//     chunk + 32r + l in registers (all loads issued up front);
//   * lanes holding the same expert in a round find each other with
//     ceil(log2(E+1)) independent __ballot_sync's (one per bit of the id);
//     the mask is kept per round and reused for ranking;
//   * up to kClusterMaxEntries entries (decode-sized batches) one kernel of
//     one thread-block cluster does everything (cluster_layout_kernel): each
//     CTA ranks its own slice of the entries (__match_any_sync peer masks,
//     per-warp counts), publishes its expert histogram in shared memory, and
//     after a cluster barrier reads its peers' histograms through distributed
//     shared memory (four peers' loads in flight at once) for the expert
//     totals and its slice's base; the CTAs share the row_src fill; no
//     workspace, and no CTA reads more than its own slice of topk_idx;
//   * beyond that, tile_hist_kernel counts each tile's experts (shared-memory
//     atomics; counts need no order) into the scratch workspace [tiles][E],
//     then assign_kernel (launched as a programmatic dependent, so its loads
//     and ballots overlap tile_hist) waits for it and sums the workspace
//     columns into the expert totals and its tile's base;
//   * assign_kernel scans the padded counts, turns per-warp histograms into
//     per-warp starting slots and gives each entry
//     slot = warp base + #lower lanes with the same expert: exactly ascending
//     (token, k) order;
//   * extra CTAs (masked layouts with row_src) only count the experts with
//     shared-memory atomics and write -1 into row_src for empty slots.
#include "ep_common.cuh"

namespace ep {
namespace {

constexpr int kRounds = 8;       // max 32-entry rounds per warp chunk
constexpr int kChunk = 32 * kRounds;
constexpr int kFillCtas = 128;
constexpr int kSumChunk = 16;    // workspace loads in flight per thread
constexpr int kSmallThreads = 1024;                     // single-tile CTA
constexpr int kTileThreads = 256;                       // multi-tile CTAs
constexpr int kSmallMax = kSmallThreads;                // 1024 entries: one round per warp
constexpr int kSelfHistMax = 4096;  // up to here every tile CTA recounts all entries itself

__host__ __device__ inline int round_up_pow2(int v, int a) { return (v + a - 1) & ~(a - 1); }

// A warp chunk, up to kRounds entries per lane: ids (invalid ones mapped to
// E), peer masks (lanes with the same id this round) and the bad-id flags.
struct Chunk {
    int ev[kRounds];
    unsigned peers[kRounds];
    unsigned bad;
};

// Issue the chunk's loads (entries past c1 read as -1).
__device__ __forceinline__ void fetch_chunk(const int32_t *__restrict__ idx, int c0, int c1,
                                            Chunk &c) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int r = 0; r < kRounds; ++r) {
        const int i = c0 + r * 32 + lane;
        c.ev[r] = i < c1 ? __ldg(idx + i) : -1;
    }
}

// Map invalid ids to E (recording bad ones) and find each round's peers.
__device__ __forceinline__ void classify_chunk(int c0, int c1, int E, int nbits, Chunk &c) {
    c.bad = 0;
#pragma unroll
    for (int r = 0; r < kRounds; ++r) {
        const int e = c.ev[r];
        if (e < -1 || e >= E) c.bad |= 1u << r;
        c.ev[r] = (e >= 0 && e < E) ? e : E;  // E = no expert
    }
#pragma unroll
    for (int r = 0; r < kRounds; ++r) {
        unsigned m = 0;
        if (c0 + r * 32 < c1) {  // warp-uniform: rounds past the chunk stay empty
            const int v = c.ev[r];
            m = kFullMask;
#pragma unroll 1
            for (int b = 0; b < nbits; ++b) {  // warp-uniform trip count; kept rolled (code size)
                const unsigned bit = (v >> b) & 1u;
                const unsigned bal = __ballot_sync(kFullMask, bit);
                m &= bit ? bal : ~bal;
            }
        }
        c.peers[r] = m;
    }
}

__device__ __forceinline__ void load_chunk(const int32_t *__restrict__ idx, int c0, int c1,
                                           int E, int nbits, Chunk &c) {
    fetch_chunk(idx, c0, c1, c);
    classify_chunk(c0, c1, E, nbits, c);
}


__device__ __forceinline__ int id_bits(int E) { return 32 - __clz(E); }  // E itself must fit

__device__ __forceinline__ void pdl_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

__global__ void __launch_bounds__(kTileThreads)
    tile_hist_kernel(const int32_t *__restrict__ idx, int TK, int E, int tile,
                     int32_t *__restrict__ ws, int32_t *__restrict__ status) {
    // First kernel of the layout, launched as a programmatic dependent: wait
    // for the previous kernel on the stream (it may have produced topk_idx,
    // and it may still read this layout's arrays) before anything else, and
    // only then let the assign kernel -- which reads topk_idx before its own
    // wait -- and dispatch start.
    pdl_wait();
    pdl_launch_dependents();
    extern __shared__ int32_t hist[];  // [E]
    for (int e = threadIdx.x; e < E; e += kTileThreads) hist[e] = 0;
    __syncthreads();
    // counts only: order does not matter, one shared-memory atomic per entry
    const int start = blockIdx.x * tile;
    const int end = min(TK, start + tile);
    for (int i = start + (int)threadIdx.x; i < end; i += kTileThreads) {
        const int e = __ldg(idx + i);
        if (e >= 0 && e < E) atomicAdd(&hist[e], 1);
    }
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += kTileThreads) ws[(size_t)blockIdx.x * E + e] = hist[e];
    // The assign kernel raises errors only after waiting for this kernel.
    if (blockIdx.x == 0 && threadIdx.x == 0) *status = EP_OK;
}

struct AssignArgs {
    const int32_t *idx;
    int TK, E, R, masked, align, cap;
    int chunk;   // entries per warp per pass (multiple of 32, <= kChunk)
    int passes;  // passes per tile
    int tile, tiles;
    int self_hist;      // tiles > 1 without the histogram kernel (see layout_plan)
    int first;          // the layout's only kernel (no tile_hist_kernel before it)
    const int32_t *ws;  // [tiles][E]; unused when tiles == 1 or self_hist
    int32_t *dst_row, *row_src, *count, *offset, *rank_rows, *status;
};

template <int NT>
__global__ void __launch_bounds__(NT) assign_kernel(AssignArgs a) {
    constexpr int kWarps = NT / 32;
    extern __shared__ int32_t sm[];
    const int E = a.E;
    const int passes = a.passes;
    int32_t *wh = sm;                         // [passes][kWarps][E]: per-warp counts, then slot bases
    int32_t *tot = wh + passes * kWarps * E;  // [E] expert histogram
    int32_t *off = tot + E;                   // [E+1] first row of each expert
    int32_t *pre = off + E + 1;               // [E] self_hist: entries before this tile
    __shared__ int32_t scan_tmp[kWarps];

    // as the first kernel: wait for the previous kernel before anything else
    // (see tile_hist_kernel); then dispatch may start loading and quantising x
    if (a.first) pdl_wait();
    pdl_launch_dependents();

    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const bool assigns = blockIdx.x < a.tiles;
    const int tile_id = blockIdx.x;
    const int start = tile_id * a.tile;
    const int end = min(a.TK, start + a.tile);
    const int nbits = id_bits(E);
    const int pass_len = kWarps * a.chunk;

    if (!assigns) {
        // Fill CTA (masked layouts with row_src): only the expert counts are
        // needed, in any order; masked offsets are e*cap, so no scan either.
        if (a.tiles == 1 || a.self_hist) {
            for (int e = threadIdx.x; e < E; e += NT) tot[e] = 0;
            __syncthreads();
            count_all<NT>(a.idx, a.TK, E, 0, tot, nullptr);
        } else {
            pdl_wait();
            for (int e = threadIdx.x; e < E; e += NT) {
                int total = 0;
                for (int b = 0; b < a.tiles; ++b) total += ld_dep(a.ws + (size_t)b * E + e);
                tot[e] = total;
            }
        }
        __syncthreads();
        for (int e = blockIdx.x + (int)gridDim.x * warp; e < E; e += (int)gridDim.x * kWarps)
            for (int r = e * a.cap + min(tot[e], a.cap) + lane; r < (e + 1) * a.cap; r += 32)
                a.row_src[r] = -1;
        return;
    }

    // single-pass tiles: the chunk's loads go out first, so that their latency
    // overlaps the zeroing (and the recount) below
    Chunk c;
    if (passes == 1)
        fetch_chunk(a.idx, start + warp * a.chunk, min(end, start + warp * a.chunk + a.chunk), c);
    for (int j = threadIdx.x; j < passes * kWarps * E; j += NT) wh[j] = 0;
    if (a.self_hist) {
        // No histogram kernel: every tile CTA recounts all entries (a few
        // shared-memory atomics per thread at these sizes): the expert totals
        // and the entries before its own tile.  Done first, so that the chunk
        // loads below find this tile's entries in L1.  Every CTA thus sees
        // every bad id and every over-full expert, so CTA 0 alone writes the
        // status word, once, and no CTA raises errors into it.
        for (int e = threadIdx.x; e < E; e += NT) tot[e] = pre[e] = 0;
        __syncthreads();
        const int bad = __syncthreads_or(count_all<NT>(a.idx, a.TK, E, start, tot, pre));
        int over = 0;
        if (a.masked)
            for (int e = threadIdx.x; e < E; e += NT) over |= tot[e] > a.cap;
        over = __syncthreads_or(over);
        if (blockIdx.x == 0 && threadIdx.x == 0)
            *a.status = bad ? EP_ERR_BAD_EXPERT_ID : over ? EP_ERR_CAPACITY : EP_OK;
    }

    __syncthreads();

    // 1. per-(pass, warp) expert histogram of this tile; chunks stay in
    //    registers for single-pass tiles (the common case), else are reloaded.
    {
        for (int p = 0; p < passes; ++p) {
            const int c0 = start + p * pass_len + warp * a.chunk;
            const int c1 = min(end, c0 + a.chunk);
            if (passes == 1)
                classify_chunk(c0, c1, E, nbits, c);
            else
                load_chunk(a.idx, c0, c1, E, nbits, c);
            int32_t *row = wh + (p * kWarps + warp) * E;
#pragma unroll
            for (int r = 0; r < kRounds; ++r) {
                const int e = c.ev[r];
                if (e < E && lane == __ffs(c.peers[r]) - 1) row[e] += __popc(c.peers[r]);
                __syncwarp();
            }
        }
    }
    // Everything below reads the histogram kernel's workspace or writes the
    // status word it resets: wait for it (a no-op without a programmatic edge).
    pdl_wait();
    if (a.tiles == 1 && blockIdx.x == 0 && threadIdx.x == 0) *a.status = EP_OK;
    __syncthreads();

    // 2. expert totals and this tile's base; per-warp counts -> starting slots
    for (int e = threadIdx.x; e < E; e += NT) {
        int total = 0, base = 0;
        if (a.self_hist) {
            total = tot[e];
            base = pre[e];
        } else if (a.tiles == 1) {
            for (int j = 0; j < passes * kWarps; ++j) total += wh[j * E + e];
        } else {
            for (int b0 = 0; b0 < a.tiles; b0 += kSumChunk) {
                int v[kSumChunk];
#pragma unroll
                for (int u = 0; u < kSumChunk; ++u)
                    v[u] = b0 + u < a.tiles ? ld_dep(a.ws + (size_t)(b0 + u) * E + e) : 0;
#pragma unroll
                for (int u = 0; u < kSumChunk; ++u) {
                    base += b0 + u < tile_id ? v[u] : 0;
                    total += v[u];
                }
            }
        }
        tot[e] = total;
        {
            int run = base;
            for (int j = 0; j < passes * kWarps; ++j) {  // (pass, warp) order = entry order
                const int cnt = wh[j * E + e];
                wh[j * E + e] = run;
                run += cnt;
            }
        }
    }
    __syncthreads();

    // 3. padded exclusive scan (contiguous) or fixed stride (masked)
    const int align = a.align, cap = a.cap, masked = a.masked;
    block_exclusive_scan<NT>(
        E, [&](int e) { return masked ? cap : round_up_pow2(tot[e], align); }, off, scan_tmp);

    if (blockIdx.x == 0) {
        for (int e = threadIdx.x; e < E; e += NT) {
            a.count[e] = tot[e];
            a.offset[e] = off[e];
        }
        if (threadIdx.x == 0) a.offset[E] = off[E];
        if (a.rank_rows) {  // one warp per rank: sum of its experts' counts
            const int per = E / a.R;
            for (int r = warp; r < a.R; r += kWarps) {
                int sum = 0;
                for (int e = r * per + lane; e < (r + 1) * per; e += 32) sum += tot[e];
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(kFullMask, sum, o);
                if (lane == 0) a.rank_rows[r] = sum;
            }
        }
    }

    // 4. stable slots: warp base + rank among lower lanes with the same expert
    {
        for (int p = 0; p < passes; ++p) {
            const int c0 = start + p * pass_len + warp * a.chunk;
            const int c1 = min(end, c0 + a.chunk);
            if (passes > 1) load_chunk(a.idx, c0, c1, E, nbits, c);
            int32_t *row = wh + (p * kWarps + warp) * E;
#pragma unroll
            for (int r = 0; r < kRounds; ++r) {
                const int i0 = c0 + r * 32;
                if (i0 >= c1) break;  // warp-uniform
                const int e = c.ev[r];
                const unsigned peers = c.peers[r];
                const int slot = e < E ? row[e] + __popc(peers & lanemask_lt()) : 0;
                __syncwarp();
                if (e < E && lane == __ffs(peers) - 1) row[e] += __popc(peers);
                __syncwarp();
                const int i = i0 + lane;
                if (i < c1) {
                    int dst = -1;
                    if (c.bad & (1u << r)) {
                        if (!a.self_hist) raise_status(a.status, EP_ERR_BAD_EXPERT_ID);
                    } else if (e < E) {
                        if (masked && slot >= cap) {
                            if (!a.self_hist) raise_status(a.status, EP_ERR_CAPACITY);
                        } else {
                            dst = off[e] + slot;
                        }
                    }
                    a.dst_row[i] = dst;
                    if (dst >= 0 && a.row_src) a.row_src[dst] = i;
                }
            }
        }
    }

    // 5. row_src = -1 on padding rows (contiguous) and empty slots (masked);
    //    fill CTAs, when present, took the other experts
    if (a.row_src) {  // one warp per expert
        for (int e = blockIdx.x + (int)gridDim.x * warp; e < E; e += (int)gridDim.x * kWarps) {
            const int r0 = off[e] + (masked ? min(tot[e], cap) : tot[e]);
            const int r1 = masked ? off[e] + cap : off[e + 1];
            for (int r = r0 + lane; r < r1; r += 32) a.row_src[r] = -1;
        }
    }
}

// ---- decode-sized batches: one thread-block cluster ----

constexpr int kClThreads = 256;          // threads per CTA of the cluster kernel
constexpr int kClWarps = kClThreads / 32;
constexpr int kClTargetPerCta = 256;     // entries per CTA aimed for (one round per warp)
constexpr int kClMaxCtas = 16;           // CTAs per cluster (16 needs the non-portable opt-in)
constexpr int kClusterMaxEntries = 16384;  // 8 CTAs of 8 rounds per warp hold it too

__device__ __forceinline__ unsigned cluster_ctarank() {
    unsigned r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ unsigned cluster_nctarank() {
    unsigned r;
    asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
    return r;
}
// All threads of every CTA of the cluster take part (uniform control flow).
__device__ __forceinline__ void cluster_arrive() {
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_arrive_relaxed() {
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// The shared-memory word that `p` names, read from the CTAs of cluster ranks
// c0 .. c0+3 (distributed shared memory), all four loads in flight at once.
// Ranks at or past csize read rank 0 and give 0.
__device__ __forceinline__ void ld_peers4(const int32_t *p, unsigned c0, unsigned csize,
                                          int32_t v[4]) {
    const uint32_t a = static_cast<uint32_t>(__cvta_generic_to_shared(p));
    const unsigned r0 = c0 < csize ? c0 : 0, r1 = c0 + 1 < csize ? c0 + 1 : 0;
    const unsigned r2 = c0 + 2 < csize ? c0 + 2 : 0, r3 = c0 + 3 < csize ? c0 + 3 : 0;
    asm volatile(
        "{\n\t.reg .b32 a0, a1, a2, a3;\n\t"
        "mapa.shared::cluster.u32 a0, %4, %5;\n\t"
        "mapa.shared::cluster.u32 a1, %4, %6;\n\t"
        "mapa.shared::cluster.u32 a2, %4, %7;\n\t"
        "mapa.shared::cluster.u32 a3, %4, %8;\n\t"
        "ld.shared::cluster.s32 %0, [a0];\n\t"
        "ld.shared::cluster.s32 %1, [a1];\n\t"
        "ld.shared::cluster.s32 %2, [a2];\n\t"
        "ld.shared::cluster.s32 %3, [a3];\n\t}"
        : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3])
        : "r"(a), "r"(r0), "r"(r1), "r"(r2), "r"(r3)
        : "memory");
#pragma unroll
    for (int j = 0; j < 4; ++j) v[j] = c0 + j < csize ? v[j] : 0;
}

// v = -1 for rows [r0, r1) of row_src; 16-byte stores where the address allows.
__device__ __forceinline__ void fill_minus_one(int32_t *row_src, int r0, int r1, int lane) {
    if (r0 >= r1) return;
    const int head = (int)((16 - (reinterpret_cast<uintptr_t>(row_src + r0) & 15)) & 15) / 4;
    const int a = min(r1, r0 + head);        // first 16-byte-aligned row (or r1)
    const int b = a + ((r1 - a) & ~3);       // end of the aligned run
    if (lane < a - r0) row_src[r0 + lane] = -1;
    const int4 m1 = make_int4(-1, -1, -1, -1);
    for (int r = a + 4 * lane; r < b; r += 128) *reinterpret_cast<int4 *>(row_src + r) = m1;
    if (lane < r1 - b) row_src[b + lane] = -1;
}

struct ClusterArgs {
    const int32_t *idx;
    int TK, E, R, masked, align, cap;
    int chunk;  // entries per warp (32 * rounds)
    int32_t *dst_row, *row_src, *count, *offset, *rank_rows, *status;
};

// Grid: one or more clusters.  Every cluster lays out all TK entries the
// same way (CTA c of a cluster owns entries [c * 8 * chunk, (c + 1) * 8 *
// chunk), warp w of it the chunk at w * chunk), so (CTA, warp, round, lane)
// order is entry order and the slot of an entry is
//   (entries of its expert in lower CTAs) + (in lower warps of its CTA)
//   + (in earlier rounds of its warp) + (in lower lanes of its round).
// Cluster 0 writes the layout arrays; the row_src fill of empty rows is
// shared by the warps of all clusters (a second cluster spreads a large
// masked fill over more SMs).
template <int ROUNDS>
__global__ void __launch_bounds__(kClThreads) cluster_layout_kernel(ClusterArgs a) {
    extern __shared__ int32_t csm[];
    const int E = a.E;
    int32_t *wh = csm;                  // [kClWarps][E] per-warp counts, then warp bases
    int32_t *hist = wh + kClWarps * E;  // [E+1] this CTA's expert counts; [E] = bad-id flag
    int32_t *tot = hist + E + 1;        // [E] expert totals
    int32_t *base = tot + E;            // [E] entries of each expert in lower CTAs
    int32_t *off = base + E;            // [E+1] first row of each expert
    __shared__ int32_t scan_tmp[kClWarps];
    __shared__ int32_t s_flags;         // bit 0: a bad id; bit 1: a masked expert over capacity

    // The layout's only kernel: wait for the previous kernel on the stream (it
    // may have produced topk_idx, and may still read these arrays) before
    // anything else; then the next kernel (dispatch) may start.
    pdl_wait();
    pdl_launch_dependents();

    const unsigned crank = cluster_ctarank(), csize = cluster_nctarank();
    const bool writer = blockIdx.x < csize;  // cluster 0
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int w0 = ((int)crank * kClWarps + warp) * a.chunk;
    const int w1 = min(a.TK, w0 + a.chunk);

    // 1. this warp's entries, all loads in flight at once; the warp zeroes
    //    its own count row meanwhile
    int ev[ROUNDS];
#pragma unroll
    for (int r = 0; r < ROUNDS; ++r) {
        const int i = w0 + r * 32 + lane;
        ev[r] = i < w1 ? __ldg(a.idx + i) : -1;
    }
    int32_t *row = wh + warp * E;
    for (int e = lane; e < E; e += 32) row[e] = 0;
    if (threadIdx.x == 0) s_flags = 0;
    __syncwarp();

    // 2. per round: peers with the same expert; rank among them; warp counts
    int rank[ROUNDS];
    int bad = 0;
#pragma unroll
    for (int r = 0; r < ROUNDS; ++r) {
        const int e0 = ev[r];
        bad |= e0 < -1 || e0 >= E;
        const int e = (e0 >= 0 && e0 < E) ? e0 : E;  // E = no expert
        ev[r] = e;
        const unsigned peers = __match_any_sync(kFullMask, e);
        const int before = e < E ? row[e] : 0;
        __syncwarp();
        if (e < E && lane == __ffs(peers) - 1) row[e] = before + __popc(peers);
        __syncwarp();
        rank[r] = before + __popc(peers & lanemask_lt());
    }
    bad = __syncthreads_or(bad);

    // 3. warp counts -> warp bases within the CTA; the CTA's histogram
    for (int e = threadIdx.x; e < E; e += kClThreads) {
        int run = 0;
#pragma unroll
        for (int w = 0; w < kClWarps; ++w) {
            const int c = wh[w * E + e];
            wh[w * E + e] = run;
            run += c;
        }
        hist[e] = run;
    }
    if (threadIdx.x == 0) hist[E] = bad;

    // 4. every CTA's histogram is visible to the cluster; totals and this
    //    CTA's base from all of them, plus the error flags
    cluster_arrive();
    cluster_wait();
    const int cap = a.cap, masked = a.masked;
    int flags = 0;
    for (int e = threadIdx.x; e < E; e += kClThreads) {
        int t = 0, b = 0;
        for (unsigned c = 0; c < csize; c += 4) {
            int v[4];
            ld_peers4(hist + e, c, csize, v);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                t += v[j];
                b += c + j < crank ? v[j] : 0;
            }
        }
        tot[e] = t;
        base[e] = b;
        if (masked && t > cap) flags |= 2;
    }
    if (threadIdx.x < csize) {
        int v[4];
        ld_peers4(hist + E, threadIdx.x, threadIdx.x + 1, v);  // peer threadIdx.x's flag
        if (v[0]) flags |= 1;
    }
    // done reading the peers (nothing to publish: relaxed); they may exit
    // once every thread of the cluster has arrived here
    cluster_arrive_relaxed();
    if (flags) atomicOr(&s_flags, flags);

    // 5. offsets: e*cap (masked) or the padded exclusive scan (contiguous)
    const int align = a.align;
    if (masked) {
        for (int e = threadIdx.x; e <= E; e += kClThreads) off[e] = e * cap;
        __syncthreads();
    } else {
        __syncthreads();
        block_exclusive_scan<kClThreads>(
            E, [&](int e) { return round_up_pow2(tot[e], align); }, off, scan_tmp);
    }

    if (writer) {
        // 6. stable slots of this warp's entries
#pragma unroll
        for (int r = 0; r < ROUNDS; ++r) {
            const int i = w0 + r * 32 + lane;
            if (i < w1) {
                const int e = ev[r];
                int dst = -1;
                if (e < E) {
                    const int slot = base[e] + row[e] + rank[r];
                    if (!(masked && slot >= cap)) dst = off[e] + slot;
                }
                a.dst_row[i] = dst;
                if (dst >= 0 && a.row_src) a.row_src[dst] = i;
            }
        }
        // 7. counts and offsets, a slice of the experts per CTA; the status
        //    word from CTA 0, the rank rows from the last CTA
        for (int e = (int)crank * kClThreads + threadIdx.x; e < E; e += (int)csize * kClThreads) {
            a.count[e] = tot[e];
            a.offset[e] = off[e];
        }
        if (crank == 0 && threadIdx.x == 0) {
            const int f = s_flags;
            *a.status = (f & 1) ? EP_ERR_BAD_EXPERT_ID : (f & 2) ? EP_ERR_CAPACITY : EP_OK;
        }
        if (crank == csize - 1) {
            if (threadIdx.x == 0) a.offset[E] = off[E];
            if (a.rank_rows) {  // one warp per rank: sum of its experts' counts
                const int per = E / a.R;
                for (int rr = warp; rr < a.R; rr += kClWarps) {
                    int sum = 0;
                    for (int e = rr * per + lane; e < (rr + 1) * per; e += 32) sum += tot[e];
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(kFullMask, sum, o);
                    if (lane == 0) a.rank_rows[rr] = sum;
                }
            }
        }
    }

    // 8. row_src = -1 on padding rows (contiguous) and empty slots (masked),
    //    one warp per expert across all clusters
    if (a.row_src) {
        const int gw = (int)blockIdx.x * kClWarps + warp, nw = (int)gridDim.x * kClWarps;
        for (int e = gw; e < E; e += nw) {
            const int r0 = off[e] + (masked ? min(tot[e], cap) : tot[e]);
            const int r1 = masked ? off[e] + cap : off[e + 1];
            fill_minus_one(a.row_src, r0, r1, lane);
        }
    }
    // no CTA leaves while a peer may still read its histogram
    cluster_wait();
}

using ClusterKernel = void (*)(ClusterArgs);

ClusterKernel cluster_kernel(int rounds) {
    switch (rounds) {
        case 1: return cluster_layout_kernel<1>;
        case 2: return cluster_layout_kernel<2>;
        case 4: return cluster_layout_kernel<4>;
        default: return cluster_layout_kernel<8>;
    }
}

}  // namespace

namespace {

// Dynamic shared memory of the cluster kernel: per-warp counts, the CTA's
// histogram (+ bad-id flag), totals, bases and offsets.
size_t cluster_smem(int E) {
    return sizeof(int32_t) * ((size_t)kClWarps * E + 4 * (size_t)E + 2);
}

// CTAs of the cluster kernel for TK entries with at most max_ctas per
// cluster, and the entries per warp (32 x a power-of-two number of rounds).
void cluster_shape(long long TK, int max_ctas, int *ctas, int *chunk) {
    long long c = (TK + kClTargetPerCta - 1) / kClTargetPerCta;
    if (c < 1) c = 1;
    if (c > max_ctas) c = max_ctas;
    int rounds = 1;
    while ((long long)rounds * 32 * kClWarps * c < TK) rounds *= 2;
    // as few CTAs as the rounds allow (fewer peers to read)
    while (c > 1 && (long long)rounds * 32 * kClWarps * (c - 1) >= TK) --c;
    *ctas = (int)c;
    *chunk = 32 * rounds;
}

// Clusters of the cluster kernel: one, or two to share a large masked
// row_src fill (the fill is bound by each SM's store rate, about 30 bytes
// per clock; more than two clusters measured slower at the DeepSeek-V3
// decode shape).
int fill_clusters(const ep_layout_t &L, int ctas) {
    if (L.kind != EP_LAYOUT_MASKED || L.row_src == nullptr) return 1;
    const long long rows = (long long)L.num_experts * L.capacity;
    return rows > (long long)ctas * 2048 ? 2 : 1;
}

// 16 CTAs per cluster where the device can co-schedule them (with the
// largest shared memory the kernel asks for), else the portable 8; once per
// device.
int max_cluster_ctas() {
    static int cached[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 8;
    if (cached[dev] == 0) {
        int best = 8;
        const size_t smem = cluster_smem(EP_MAX_EXPERTS);
        const ClusterKernel k = cluster_kernel(8);
        if (allow_dynamic_smem(k, smem) == cudaSuccess &&
            cudaFuncSetAttribute(k, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) ==
                cudaSuccess) {
            cudaLaunchConfig_t cfg = {};
            cfg.gridDim = dim3(kClMaxCtas);
            cfg.blockDim = dim3(kClThreads);
            cfg.dynamicSmemBytes = smem;
            cudaLaunchAttribute attr[1];
            attr[0].id = cudaLaunchAttributeClusterDimension;
            attr[0].val.clusterDim.x = kClMaxCtas;
            attr[0].val.clusterDim.y = 1;
            attr[0].val.clusterDim.z = 1;
            cfg.attrs = attr;
            cfg.numAttrs = 1;
            int n = 0;
            if (cudaOccupancyMaxActiveClusters(&n, k, &cfg) == cudaSuccess &&
                n >= 1)
                best = kClMaxCtas;
        }
        cudaGetLastError();  // a refused query leaves no error behind
        cached[dev] = best;
    }
    return cached[dev];
}

}  // namespace

LayoutPlan layout_plan(const ep_layout_t &L) {
    LayoutPlan p{};
    const long long TK = (long long)L.num_tokens * L.num_topk;
    int warps;
    if (TK <= kClusterMaxEntries) {
        // one cluster (its CTA count is chosen at launch: 8 or 16 at most)
        int ctas, chunk;
        cluster_shape(TK, kClMaxCtas, &ctas, &chunk);
        p.cluster = true;
        p.threads = kClThreads;
        p.tiles = ctas;
        p.grid = ctas;
        p.passes = 1;
        p.chunk = chunk;
        p.tile = chunk * kClWarps;
        p.self_hist = false;
        p.smem = cluster_smem(L.num_experts);
        p.ws_bytes = 0;
        return p;
    }
    if (TK <= kSmallMax) {
        // one 1024-thread CTA, one 32-entry round per warp
        p.threads = kSmallThreads;
        warps = kSmallThreads / 32;
        p.tiles = 1;
        p.passes = 1;
        p.chunk = 32;
        p.tile = p.chunk * warps;
    } else {
        // 256-thread tiles: 4 rounds per warp (1024 entries) spread mid-size
        // inputs over more SMs, 8 rounds (2048) for large ones; beyond 128
        // tiles the tile grows in whole passes, which bounds the workspace
        p.threads = kTileThreads;
        warps = kTileThreads / 32;
        p.chunk = TK <= 32768 ? kChunk / 2 : kChunk;
        const long long pass_len = (long long)warps * p.chunk;
        long long tiles = (TK + pass_len - 1) / pass_len;
        p.passes = 1;
        if (tiles > 128) {
            p.passes = (int)((tiles + 127) / 128);
            tiles = (TK + pass_len * p.passes - 1) / (pass_len * p.passes);
        }
        p.tiles = (int)tiles;
        p.tile = (int)pass_len * p.passes;
    }
    // few tiles: one kernel, each tile CTA recounting every entry, instead of
    // a histogram kernel and a workspace (a kernel boundary saved on decode)
    p.self_hist = p.tiles > 1 && TK <= kSelfHistMax;
    const bool fill = L.kind == EP_LAYOUT_MASKED && L.row_src != nullptr;
    p.grid = p.tiles;
    if (fill && p.grid < kFillCtas) p.grid = L.num_experts < kFillCtas ? L.num_experts : kFillCtas;
    if (p.grid < p.tiles) p.grid = p.tiles;
    p.smem = sizeof(int32_t) * ((size_t)p.passes * warps * L.num_experts +
                                (p.self_hist ? 3 : 2) * (size_t)L.num_experts + 1);
    p.ws_bytes = p.tiles > 1 && !p.self_hist ? sizeof(int32_t) * (size_t)p.tiles * L.num_experts : 0;
    return p;
}

cudaError_t launch_layout(const int32_t *topk_idx, const ep_layout_t &L, int32_t *workspace,
                          cudaStream_t stream) {
    const LayoutPlan p = layout_plan(L);
    const int TK = L.num_tokens * L.num_topk;
    const int E = L.num_experts;
    if (p.cluster) {
        ClusterArgs c;
        c.idx = topk_idx;
        c.TK = TK;
        c.E = E;
        c.R = L.num_ranks;
        c.masked = L.kind == EP_LAYOUT_MASKED;
        c.align = c.masked ? 1 : L.align;
        c.cap = c.masked ? L.capacity : 0;
        int ctas;
        cluster_shape(TK, max_cluster_ctas(), &ctas, &c.chunk);
        const int nclusters = fill_clusters(L, ctas);
        c.dst_row = L.dst_row;
        c.row_src = L.row_src;
        c.count = L.expert_count;
        c.offset = L.expert_offset;
        c.rank_rows = L.rank_rows;
        c.status = L.status;
        const ClusterKernel k = cluster_kernel(c.chunk / 32);
        const size_t smem = cluster_smem(E);
        cudaError_t err = allow_dynamic_smem(k, smem);
        if (err != cudaSuccess) return err;
        if (ctas > 8) {
            err = cudaFuncSetAttribute(k, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
            if (err != cudaSuccess) return err;
        }
        // the layout's only kernel: programmatic, waiting for the previous kernel first
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(ctas * nclusters);
        cfg.blockDim = dim3(kClThreads);
        cfg.dynamicSmemBytes = smem;
        cfg.stream = stream;
        cudaLaunchAttribute attr[2];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = ctas;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[1].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 2;
        return cudaLaunchKernelEx(&cfg, k, c);
    }
    AssignArgs a;
    a.idx = topk_idx;
    a.TK = TK;
    a.E = E;
    a.R = L.num_ranks;
    a.masked = L.kind == EP_LAYOUT_MASKED;
    a.align = a.masked ? 1 : L.align;
    a.cap = a.masked ? L.capacity : 0;
    a.chunk = p.chunk;
    a.passes = p.passes;
    a.tile = p.tile;
    a.tiles = p.tiles;
    a.self_hist = p.self_hist;
    a.first = p.threads == kSmallThreads || p.self_hist;
    a.ws = workspace;
    a.dst_row = L.dst_row;
    a.row_src = L.row_src;
    a.count = L.expert_count;
    a.offset = L.expert_offset;
    a.rank_rows = L.rank_rows;
    a.status = L.status;
    cudaError_t err;
    if (p.threads == kSmallThreads) {
        err = allow_dynamic_smem(assign_kernel<kSmallThreads>, p.smem);
        if (err != cudaSuccess) return err;
        // the only kernel: programmatic, waiting for the previous kernel first
        return launch_kernel(assign_kernel<kSmallThreads>, p.grid, kSmallThreads, p.smem, stream,
                             true, a);
    }
    if (p.self_hist) {  // the only kernel: programmatic, waiting for the previous kernel first
        err = allow_dynamic_smem(assign_kernel<kTileThreads>, p.smem);
        if (err != cudaSuccess) return err;
        return launch_kernel(assign_kernel<kTileThreads>, p.grid, kTileThreads, p.smem, stream,
                             true, a);
    }
    err = launch_kernel(tile_hist_kernel, p.tiles, kTileThreads, sizeof(int32_t) * E, stream,
                        true, topk_idx, TK, E, p.tile, workspace, L.status);
    if (err != cudaSuccess) return err;
    err = allow_dynamic_smem(assign_kernel<kTileThreads>, p.smem);
    if (err != cudaSuccess) return err;
    return launch_kernel(assign_kernel<kTileThreads>, p.grid, kTileThreads, p.smem, stream, true,
                         a);
}

}  // namespace ep
