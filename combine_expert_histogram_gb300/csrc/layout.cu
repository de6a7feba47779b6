// ep_layout kernels: expert histogram, padded exclusive scan, stable slots.
//
// The layout step that DeepEP V2's dispatch performs internally ("infers the
// layout from topk_idx", SGLang PR "moe: add DeepEP V2 ElasticBuffer support
// to MoE token dispatcher", section "Motivation"), for the contiguous
// (prefill) and masked (decode) layouts of SGLang PR "[Feature] Add DeepEPv2
// (ElasticBuffer) MoE A2A backend", section "Supported scope".
//
// Design (deterministic, no global atomics on slot order; latency-bound, so
// the goal is short dependency chains and many warps).  In both paths lanes
// holding the same expert in a round of 32 entries find each other (a peer
// mask), and an entry's slot is the number of entries of its expert before
// it: in lower CTAs or tiles, in lower warps, in earlier rounds and in lower
// lanes -- exactly ascending (token, k) order.
//
//   * Up to 16384 entries (decode-sized batches): one kernel of 2-4
//     thread-block clusters (cluster_layout_kernel; its body is in
//     cluster_layout.cuh).  Each CTA of the first cluster ranks its own slice of the entries with
//     per-warp counts and pushes its expert histogram into every peer's
//     shared memory (one bulk copy per peer through distributed shared
//     memory, completing on the peer's mbarrier); each CTA sums the blocks it
//     received for the expert totals and its slice's base.  No workspace, and
//     no CTA reads more than its own slice of topk_idx.  This ranking
//     cluster writes the slots; 1-3 more clusters that only count write the
//     counts, offsets and status and share the row_src fill.  Peer masks from
//     one ballot per bit of the id.
//   * Beyond that: tile_hist_kernel counts each tile's experts (shared-memory
//     atomics; counts need no order) into the workspace [tiles][E]; then
//     assign_kernel, a programmatic dependent whose loads and match masks
//     overlap tile_hist, waits for it, sums the workspace columns into the
//     expert totals and its tile's base, scans the padded counts, turns
//     per-warp histograms into per-warp starting slots and writes the slots.
//     Warp w of a tile's CTA owns a contiguous chunk of up to 256 entries,
//     lane l holding entries chunk + 32r + l in registers (all loads issued
//     up front).  Peer masks from one __match_any_sync per round, which
//     replaced one __ballot_sync per bit of the id here (601 k -> 384 k warp
//     instructions, 14.0 -> 11.4 us for 65536 entries).  Extra CTAs of masked layouts with row_src only
//     sum the expert totals and write -1 into row_src for empty slots.
#include <stdlib.h>

#include <mutex>

#include "cluster_layout.cuh"

namespace ep {
namespace {

constexpr int kRounds = 8;       // max 32-entry rounds per warp chunk
constexpr int kChunk = 32 * kRounds;
constexpr int kFillCtas = 128;
constexpr int kSumChunk = 16;    // workspace loads in flight per thread
constexpr int kTileThreads = 256;  // threads of the tile CTAs

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
__device__ __forceinline__ void classify_chunk(int c0, int c1, int E, Chunk &c) {
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
        if (c0 + r * 32 < c1)  // warp-uniform: rounds past the chunk stay empty
            m = __match_any_sync(kFullMask, c.ev[r]);
        c.peers[r] = m;
    }
}

__device__ __forceinline__ void load_chunk(const int32_t *__restrict__ idx, int c0, int c1,
                                           int E, Chunk &c) {
    fetch_chunk(idx, c0, c1, c);
    classify_chunk(c0, c1, E, c);
}

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
    const int32_t *ws;  // [tiles][E] per-tile histograms of tile_hist_kernel
    int32_t *dst_row, *row_src, *count, *offset, *rank_rows, *status;
};

// Launched as a programmatic dependent of tile_hist_kernel: the tile's loads
// and ballots run before griddepcontrol.wait, everything that reads the
// workspace or touches the status word after it.
__global__ void __launch_bounds__(kTileThreads) assign_kernel(AssignArgs a) {
    constexpr int NT = kTileThreads, kWarps = NT / 32;
    extern __shared__ int32_t sm[];
    const int E = a.E;
    const int passes = a.passes;
    int32_t *wh = sm;                         // [passes][kWarps][E]: per-warp counts, then slot bases
    int32_t *tot = wh + passes * kWarps * E;  // [E] expert histogram
    int32_t *off = tot + E;                   // [E+1] first row of each expert
    __shared__ int32_t scan_tmp[kWarps];

    pdl_launch_dependents();  // dispatch may start loading and quantising x

    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const bool assigns = blockIdx.x < a.tiles;
    const int tile_id = blockIdx.x;
    const int start = tile_id * a.tile;
    const int end = min(a.TK, start + a.tile);
    const int pass_len = kWarps * a.chunk;

    if (!assigns) {
        // Fill CTA (masked layouts with row_src): only the expert totals are
        // needed; masked offsets are e*cap, so no scan either.
        pdl_wait();
        for (int e = threadIdx.x; e < E; e += NT) {
            int total = 0;
            for (int b = 0; b < a.tiles; ++b) total += ld_dep(a.ws + (size_t)b * E + e);
            tot[e] = total;
        }
        __syncthreads();
        for (int e = blockIdx.x + (int)gridDim.x * warp; e < E; e += (int)gridDim.x * kWarps)
            for (int r = e * a.cap + min(tot[e], a.cap) + lane; r < (e + 1) * a.cap; r += 32)
                a.row_src[r] = -1;
        return;
    }

    // single-pass tiles: the chunk's loads go out first, so that their latency
    // overlaps the zeroing below
    Chunk c;
    if (passes == 1)
        fetch_chunk(a.idx, start + warp * a.chunk, min(end, start + warp * a.chunk + a.chunk), c);
    for (int j = threadIdx.x; j < passes * kWarps * E; j += NT) wh[j] = 0;
    __syncthreads();

    // 1. per-(pass, warp) expert histogram of this tile; chunks stay in
    //    registers for single-pass tiles (the common case), else are reloaded.
    for (int p = 0; p < passes; ++p) {
        const int c0 = start + p * pass_len + warp * a.chunk;
        const int c1 = min(end, c0 + a.chunk);
        if (passes == 1)
            classify_chunk(c0, c1, E, c);
        else
            load_chunk(a.idx, c0, c1, E, c);
        int32_t *row = wh + (p * kWarps + warp) * E;
#pragma unroll
        for (int r = 0; r < kRounds; ++r) {
            const int e = c.ev[r];
            if (e < E && lane == __ffs(c.peers[r]) - 1) row[e] += __popc(c.peers[r]);
            __syncwarp();
        }
    }
    // Everything below reads the histogram kernel's workspace or raises into
    // the status word it resets: wait for it.
    pdl_wait();
    __syncthreads();

    // 2. expert totals and this tile's base; per-warp counts -> starting slots
    for (int e = threadIdx.x; e < E; e += NT) {
        int total = 0, base = 0;
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
        tot[e] = total;
        int run = base;
        for (int j = 0; j < passes * kWarps; ++j) {  // (pass, warp) order = entry order
            const int cnt = wh[j * E + e];
            wh[j * E + e] = run;
            run += cnt;
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
    for (int p = 0; p < passes; ++p) {
        const int c0 = start + p * pass_len + warp * a.chunk;
        const int c1 = min(end, c0 + a.chunk);
        if (passes > 1) load_chunk(a.idx, c0, c1, E, c);
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
                    raise_status(a.status, EP_ERR_BAD_EXPERT_ID);
                } else if (e < E) {
                    if (masked && slot >= cap)
                        raise_status(a.status, EP_ERR_CAPACITY);
                    else
                        dst = off[e] + slot;
                }
                a.dst_row[i] = dst;
                if (dst >= 0 && a.row_src) a.row_src[dst] = i;
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

// ---- decode-sized batches: thread-block clusters (cluster_layout.cuh) ----

// Cluster 0 ranks and writes the slots; the other clusters write the counts,
// offsets, status and rank rows and fill row_src.
template <int ROUNDS>
__global__ void __launch_bounds__(cl::kClThreads) cluster_layout_kernel(cl::ClusterArgs a) {
    extern __shared__ __align__(16) int32_t csm[];
    // The layout's only kernel: wait for the previous kernel on the stream (it
    // may have produced topk_idx, and may still read these arrays) before
    // anything else; then the next kernel (dispatch) may start.
    pdl_wait();
    pdl_launch_dependents();
    if (blockIdx.x < cl::cluster_nctarank())
        cl::cluster_layout_body<ROUNDS, true>(a, csm);
    else
        cl::cluster_layout_body<ROUNDS, false>(a, csm);
}

using ClusterKernel = void (*)(cl::ClusterArgs);

ClusterKernel cluster_kernel(int rounds) {
    switch (rounds) {
        case 1: return cluster_layout_kernel<1>;
        case 2: return cluster_layout_kernel<2>;
        case 4: return cluster_layout_kernel<4>;
        default: return cluster_layout_kernel<8>;
    }
}

}  // namespace

namespace cl {

// EP_MAX_CLUSTER_CTAS=8 caps the cluster at the portable size (for a device
// partition that cannot place 16 co-scheduled CTAs, or to check that
// configuration).  The two sizes are the only ones used: any value below 16
// counts as 8 (the kernel's rounds per warp allow at most 8 x 8 x 256
// entries on 8 CTAs, so no fewer).
int cluster_ctas_cap() {
    static const int cap = [] {
        const char *v = getenv("EP_MAX_CLUSTER_CTAS");
        const int n = v ? atoi(v) : kClMaxCtas;
        return n < kClMaxCtas ? 8 : kClMaxCtas;
    }();
    return cap;
}

int max_cluster_ctas(const void *func, size_t smem) {
    struct Entry {
        const void *func;
        int dev;
        size_t smem;
        int best;
    };
    static Entry cache[32];
    static int used = 0;
    static std::mutex mu;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 8;
    std::lock_guard<std::mutex> lock(mu);
    for (int i = 0; i < used; ++i)
        if (cache[i].func == func && cache[i].dev == dev && cache[i].smem == smem)
            return cache[i].best;
    int best = 8;
    cudaFuncAttributes fa;
    bool ok = cudaFuncGetAttributes(&fa, func) == cudaSuccess;
    if (ok && smem + fa.sharedSizeBytes > 48 * 1024)
        ok = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) ==
             cudaSuccess;
    if (ok && cudaFuncSetAttribute(func, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) ==
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
        if (cudaOccupancyMaxActiveClusters(&n, func, &cfg) == cudaSuccess && n >= 1)
            best = kClMaxCtas;
    }
    cudaGetLastError();  // a refused query leaves no error behind
    if (best > cluster_ctas_cap()) best = cluster_ctas_cap();
    if (used < 32) cache[used++] = Entry{func, dev, smem, best};
    return best;
}

}  // namespace cl

// Self-test of the cluster exchange's bounded wait: two CTAs of one cluster
// initialise their barriers, meet at the cluster barrier and each wait for
// 16 bytes that no peer sends (no copy is issued, so nothing can land after
// the CTAs exit); each wait must give up after `limit` SM clocks, the CTAs
// must still meet at the final cluster barrier, and the kernel must report
// EP_ERR_TIMEOUT -- the same sequence as the layout's exchange.
__global__ void __launch_bounds__(cl::kClThreads) cluster_wait_selftest_kernel(int32_t *status, long long limit) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        mbar_init_fence();
    }
    cl::cluster_arrive_relaxed();
    __syncthreads();
    cl::cluster_wait();
    if (threadIdx.x == 0)
        asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], 16;" ::"r"(smem_addr(&bar))
                     : "memory");
    const bool ok = mbar_wait(&bar, 0, nullptr, limit);
    cl::cluster_arrive_relaxed();
    if (__syncthreads_or(!ok) && threadIdx.x == 0) raise_status(status, EP_ERR_TIMEOUT);
    cl::cluster_wait();
}

cudaError_t launch_cluster_wait_selftest(int32_t *status, long long limit_clocks,
                                         cudaStream_t stream) {
    return cl::launch_clusters(cluster_wait_selftest_kernel, 2, 1, 0, stream, false, status,
                               limit_clocks);
}

LayoutPlan layout_plan(const ep_layout_t &L) {
    LayoutPlan p{};
    const long long TK = (long long)L.num_tokens * L.num_topk;
    int warps;
    if (TK <= cl::kClusterMaxEntries) {
        // clusters of up to 16 CTAs (the count is chosen at launch: 8 or 16 at most)
        int ctas, chunk;
        cl::cluster_shape(TK, cl::kClMaxCtas, &ctas, &chunk);
        p.cluster = true;
        p.threads = cl::kClThreads;
        p.tiles = ctas;
        p.grid = ctas;
        p.passes = 1;
        p.chunk = chunk;
        p.tile = chunk * cl::kClWarps;
        p.smem = cl::cluster_smem(L.num_experts);
        p.ws_bytes = 0;
        return p;
    }
    // 256-thread tiles (at least 9 of them beyond the cluster kernel's range):
    // 4 rounds per warp (1024 entries) up to 32768 entries, 8 rounds (2048)
    // above; beyond 128 tiles the tile grows in whole passes, which bounds
    // the workspace
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
    const bool fill = L.kind == EP_LAYOUT_MASKED && L.row_src != nullptr;
    p.grid = p.tiles;
    if (fill && p.grid < kFillCtas) p.grid = L.num_experts < kFillCtas ? L.num_experts : kFillCtas;
    if (p.grid < p.tiles) p.grid = p.tiles;
    p.smem = sizeof(int32_t) * ((size_t)p.passes * warps * L.num_experts + 2 * (size_t)L.num_experts + 1);
    p.ws_bytes = sizeof(int32_t) * (size_t)p.tiles * L.num_experts;
    return p;
}

cudaError_t launch_layout(const int32_t *topk_idx, const ep_layout_t &L, int32_t *workspace,
                          cudaStream_t stream) {
    const LayoutPlan p = layout_plan(L);
    const int TK = L.num_tokens * L.num_topk;
    const int E = L.num_experts;
    if (p.cluster) {
        const ClusterKernel probe = cluster_kernel(8);
        const int max_ctas =
            cl::max_cluster_ctas(reinterpret_cast<const void *>(probe), cl::cluster_smem(EP_MAX_EXPERTS));
        int ctas, chunk;
        cl::cluster_shape(TK, max_ctas, &ctas, &chunk);
        const cl::ClusterArgs c = cl::cluster_args(topk_idx, L, chunk);
        // the layout's only kernel: programmatic, waiting for the previous kernel first
        const int clusters = cl::fill_clusters(L, ctas);
        return cl::launch_clusters(cluster_kernel(chunk / 32), ctas, clusters,
                                   cl::cluster_smem(E), stream, true, c);
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
    a.ws = workspace;
    a.dst_row = L.dst_row;
    a.row_src = L.row_src;
    a.count = L.expert_count;
    a.offset = L.expert_offset;
    a.rank_rows = L.rank_rows;
    a.status = L.status;
    cudaError_t err;
    err = launch_kernel(tile_hist_kernel, p.tiles, kTileThreads, sizeof(int32_t) * E, stream,
                        true, topk_idx, TK, E, p.tile, workspace, L.status);
    if (err != cudaSuccess) return err;
    err = allow_dynamic_smem(assign_kernel, p.smem);
    if (err != cudaSuccess) return err;
    return launch_kernel(assign_kernel, p.grid, kTileThreads, p.smem, stream, true, a);
}

}  // namespace ep
