// ep_layout kernels: expert histogram, padded exclusive scan, stable slots.
//
// The layout step that DeepEP V2's dispatch performs internally ("infers the
// layout from topk_idx", SGLang PR "moe: add DeepEP V2 ElasticBuffer support
// to MoE token dispatcher", section "Motivation"), for the contiguous
// (prefill) and masked (decode) layouts of SGLang PR "[Feature] Add DeepEPv2
// (ElasticBuffer) MoE A2A backend", section "Supported scope".
//
// Design (deterministic, no global atomics on slot order; latency-bound, so
// the goal is short dependency chains and every SM busy):
//   * the T*K entries are cut into tiles of 2048 entries (more for huge
//     inputs), one CTA of 256 threads per tile; warp w owns a contiguous
//     chunk of its tile and lane l holds entries chunk + 32r + l, r < rounds,
//     in registers (all loads issued up front);
//   * lanes holding the same expert in a round find each other with
//     ceil(log2(E+1)) independent __ballot_sync's (one per bit of the id);
//     the mask is kept per round and reused for ranking;
//   * tile_hist_kernel (only with >= 2 tiles) writes each tile's expert
//     histogram to the scratch workspace [tiles][E];
//   * assign_kernel: every CTA sums the workspace columns (independent L2
//     loads) into the expert totals and its tile's base, scans the padded
//     counts, turns per-warp histograms into per-warp starting slots, and
//     gives each entry slot = warp base + #lower lanes with the same expert.
//     That order is exactly ascending (token, k);
//   * extra CTAs (masked layouts with row_src) only write -1 into row_src for
//     empty slots.
#include "ep_common.cuh"

namespace ep {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kRounds = 8;                    // 32-entry rounds per warp chunk
constexpr int kTile = kThreads * kRounds;     // 2048 entries
constexpr int kMaxBits = 11;                  // ids 0..1024 (1024 = "no expert")
constexpr int kFillCtas = 128;
constexpr int kSumChunk = 16;                 // workspace loads in flight per thread

__host__ __device__ inline int round_up_pow2(int v, int a) { return (v + a - 1) & ~(a - 1); }

// A warp chunk, kRounds entries per lane: ids (invalid ones mapped to E),
// peer masks (lanes with the same id this round) and the bad-id flags.
struct Chunk {
    int ev[kRounds];
    unsigned peers[kRounds];
    unsigned bad;
};

__device__ __forceinline__ void load_chunk(const int32_t *__restrict__ idx, int c0, int c1,
                                           int E, int nbits, Chunk &c) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int r = 0; r < kRounds; ++r) {
        const int i = c0 + r * 32 + lane;
        c.ev[r] = i < c1 ? __ldg(idx + i) : -1;
    }
    c.bad = 0;
#pragma unroll
    for (int r = 0; r < kRounds; ++r) {
        const int e = c.ev[r];
        if (e < -1 || e >= E) c.bad |= 1u << r;
        c.ev[r] = (e >= 0 && e < E) ? e : E;  // E = no expert
    }
#pragma unroll
    for (int r = 0; r < kRounds; ++r) {
        const int v = c.ev[r];
        unsigned m = kFullMask;
#pragma unroll
        for (int b = 0; b < kMaxBits; ++b) {
            if (b < nbits) {  // warp-uniform
                const unsigned bit = (v >> b) & 1u;
                const unsigned bal = __ballot_sync(kFullMask, bit);
                m &= bit ? bal : ~bal;
            }
        }
        c.peers[r] = m;
    }
}

__device__ __forceinline__ int id_bits(int E) { return 32 - __clz(E); }  // E itself must fit

__global__ void __launch_bounds__(kThreads)
    tile_hist_kernel(const int32_t *__restrict__ idx, int TK, int E, int tile,
                     int32_t *__restrict__ ws, int32_t *__restrict__ status) {
    extern __shared__ int32_t hist[];  // [E]
    for (int e = threadIdx.x; e < E; e += kThreads) hist[e] = 0;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int start = blockIdx.x * tile;
    const int end = min(TK, start + tile);
    Chunk c;
    __syncthreads();  // hist zeroed
    // tiles larger than kTile (huge inputs) are walked in kTile-sized passes
    for (int base = start; base < end; base += kTile) {  // block-uniform
        const int c0 = base + warp * kRounds * 32;
        const int c1 = min(end, c0 + kRounds * 32);
        load_chunk(idx, c0, c1, E, id_bits(E), c);
#pragma unroll
        for (int r = 0; r < kRounds; ++r) {
            const int e = c.ev[r];
            if (e < E && lane == __ffs(c.peers[r]) - 1) atomicAdd(&hist[e], __popc(c.peers[r]));
        }
    }
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += kThreads) ws[(size_t)blockIdx.x * E + e] = hist[e];
    // The assign kernel runs after this one on the stream and raises errors.
    if (blockIdx.x == 0 && threadIdx.x == 0) *status = EP_OK;
}

struct AssignArgs {
    const int32_t *idx;
    int TK, E, R, masked, align, cap;
    int tile, tiles;
    const int32_t *ws;  // [tiles][E]; unused when tiles == 1
    int32_t *dst_row, *row_src, *count, *offset, *rank_rows, *status;
};

__global__ void __launch_bounds__(kThreads) assign_kernel(AssignArgs a) {
    extern __shared__ int32_t sm[];
    const int E = a.E;
    int32_t *wh = sm;                  // [passes][kWarps][E]: per-warp counts, then slot bases
    const int passes = a.tile / kTile;
    int32_t *tot = wh + passes * kWarps * E;  // [E] expert histogram
    int32_t *off = tot + E;                   // [E+1] first row of each expert
    __shared__ int32_t scan_tmp[kWarps];

    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const bool assigns = blockIdx.x < a.tiles;
    const int tile_id = assigns ? blockIdx.x : 0;
    const int start = tile_id * a.tile;
    const int end = min(a.TK, start + a.tile);
    const bool need_hist = assigns || a.tiles == 1;
    const int nbits = id_bits(E);

    // With one tile this is the only layout kernel: reset the status word
    // before any error of this CTA is raised (ordered by the barriers below).
    if (a.tiles == 1 && blockIdx.x == 0 && threadIdx.x == 0) *a.status = EP_OK;
    for (int j = threadIdx.x; j < passes * kWarps * E; j += kThreads) wh[j] = 0;
    __syncthreads();

    // 1. per-(pass, warp) expert histogram of this tile; chunks stay in registers
    //    only for single-pass tiles (the common case), else they are reloaded.
    Chunk c;
    if (need_hist) {
        for (int p = 0; p < passes; ++p) {
            const int c0 = start + p * kTile + warp * kRounds * 32;
            const int c1 = min(end, c0 + kRounds * 32);
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
    __syncthreads();

    // 2. expert totals and this tile's base; per-warp counts -> starting slots
    for (int e = threadIdx.x; e < E; e += kThreads) {
        int total = 0, base = 0;
        if (a.tiles == 1) {
            for (int j = 0; j < passes * kWarps; ++j) total += wh[j * E + e];
        } else {
            for (int b0 = 0; b0 < a.tiles; b0 += kSumChunk) {
                int v[kSumChunk];
#pragma unroll
                for (int u = 0; u < kSumChunk; ++u)
                    v[u] = b0 + u < a.tiles ? __ldcg(a.ws + (size_t)(b0 + u) * E + e) : 0;
#pragma unroll
                for (int u = 0; u < kSumChunk; ++u) {
                    base += b0 + u < tile_id ? v[u] : 0;
                    total += v[u];
                }
            }
        }
        tot[e] = total;
        if (assigns) {
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
    block_exclusive_scan<kThreads>(
        E, [&](int e) { return masked ? cap : round_up_pow2(tot[e], align); }, off, scan_tmp);

    if (blockIdx.x == 0) {
        for (int e = threadIdx.x; e < E; e += kThreads) {
            a.count[e] = tot[e];
            a.offset[e] = off[e];
        }
        if (threadIdx.x == 0) a.offset[E] = off[E];
        if (a.rank_rows) {
            const int per = E / a.R;
            for (int r = threadIdx.x; r < a.R; r += kThreads) {
                int s = 0;
                for (int e = r * per; e < (r + 1) * per; ++e) s += tot[e];
                a.rank_rows[r] = s;
            }
        }
    }

    // 4. stable slots: warp base + rank among lower lanes with the same expert
    if (assigns) {
        for (int p = 0; p < passes; ++p) {
            const int c0 = start + p * kTile + warp * kRounds * 32;
            const int c1 = min(end, c0 + kRounds * 32);
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
    }

    // 5. row_src = -1 on padding rows (contiguous) and empty slots (masked)
    if (a.row_src) {
        for (int e = blockIdx.x; e < E; e += gridDim.x) {
            const int r0 = off[e] + (masked ? min(tot[e], cap) : tot[e]);
            const int r1 = masked ? off[e] + cap : off[e + 1];
            for (int r = r0 + (int)threadIdx.x; r < r1; r += kThreads) a.row_src[r] = -1;
        }
    }
}

}  // namespace

LayoutPlan layout_plan(const ep_layout_t &L) {
    LayoutPlan p{};
    const long long TK = (long long)L.num_tokens * L.num_topk;
    // tiles of kTile entries; inputs beyond 128 tiles grow the tile by whole
    // kTile passes instead, which bounds the workspace and the column sums
    long long tiles = (TK + kTile - 1) / kTile;
    if (tiles < 1) tiles = 1;
    int passes = 1;
    if (tiles > 128) {
        passes = (int)((tiles + 127) / 128);
        tiles = (TK + (long long)kTile * passes - 1) / ((long long)kTile * passes);
    }
    p.tiles = (int)tiles;
    p.tile = kTile * passes;
    const bool fill = L.kind == EP_LAYOUT_MASKED && L.row_src != nullptr;
    p.grid = p.tiles;
    if (fill && p.grid < kFillCtas) p.grid = L.num_experts < kFillCtas ? L.num_experts : kFillCtas;
    if (p.grid < p.tiles) p.grid = p.tiles;
    p.smem = sizeof(int32_t) * ((size_t)passes * kWarps * L.num_experts + 2 * (size_t)L.num_experts + 1);
    p.ws_bytes = p.tiles > 1 ? sizeof(int32_t) * (size_t)p.tiles * L.num_experts : 0;
    return p;
}

cudaError_t launch_layout(const int32_t *topk_idx, const ep_layout_t &L, int32_t *workspace,
                          cudaStream_t stream) {
    const LayoutPlan p = layout_plan(L);
    const int TK = L.num_tokens * L.num_topk;
    const int E = L.num_experts;
    if (p.tiles > 1) {
        tile_hist_kernel<<<p.tiles, kThreads, sizeof(int32_t) * E, stream>>>(
            topk_idx, TK, E, p.tile, workspace, L.status);
        cudaError_t err = cudaGetLastError();
        if (err != cudaSuccess) return err;
    }
    if (p.smem > 48 * 1024) {
        cudaError_t err = cudaFuncSetAttribute(
            assign_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)p.smem);
        if (err != cudaSuccess) return err;
    }
    AssignArgs a;
    a.idx = topk_idx;
    a.TK = TK;
    a.E = E;
    a.R = L.num_ranks;
    a.masked = L.kind == EP_LAYOUT_MASKED;
    a.align = a.masked ? 1 : L.align;
    a.cap = a.masked ? L.capacity : 0;
    a.tile = p.tile;
    a.tiles = p.tiles;
    a.ws = workspace;
    a.dst_row = L.dst_row;
    a.row_src = L.row_src;
    a.count = L.expert_count;
    a.offset = L.expert_offset;
    a.rank_rows = L.rank_rows;
    a.status = L.status;
    assign_kernel<<<p.grid, kThreads, p.smem, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace ep
