// ep_layout kernels: expert histogram, padded exclusive scan, stable slots.
//
// The layout step that DeepEP V2's dispatch performs internally ("infers the
// layout from topk_idx", SGLang PR "moe: add DeepEP V2 ElasticBuffer support
// to MoE token dispatcher", section "Motivation"), for the contiguous
// (prefill) and masked (decode) layouts of SGLang PR "[Feature] Add DeepEPv2
// (ElasticBuffer) MoE A2A backend", section "Supported scope".
//
// Design (deterministic, no global atomics on slot order):
//   * the T*K entries are cut into tiles of <= 8192 entries, one CTA of 512
//     threads each; every warp owns a contiguous chunk of its tile and keeps
//     the chunk's ids in registers (one load per lane per 32 entries);
//   * tile_hist_kernel (only when there are >= 2 tiles) writes each tile's
//     expert histogram to the scratch workspace [tiles][E];
//   * assign_kernel: every CTA rebuilds the totals and its tile's base per
//     expert from the workspace (tiles x E ints from L2), scans the padded
//     counts, then ranks its entries: per-warp histograms give each warp's
//     starting slot per expert, and inside a warp __match_any_sync groups the
//     lanes holding the same expert, so a lane's slot is its warp base plus
//     the number of lower lanes in its group.  That order is exactly
//     ascending (token, k);
//   * extra CTAs (masked layouts) only write -1 into row_src for empty slots.
#include "ep_common.cuh"

namespace ep {
namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kRounds = 16;                   // 32-entry rounds per warp chunk
constexpr int kMaxTile = kThreads * kRounds;  // 8192 entries
constexpr int kFillCtas = 128;

__host__ __device__ inline int round_up_pow2(int v, int a) { return (v + a - 1) & ~(a - 1); }

// Load a warp chunk's ids: lane l gets entries c0 + 32*r + l, r < rounds.
// Invalid ids (outside [0, E)) and entries past c1 read as -1; `bad` flags
// rounds whose entry exists but holds an id outside [-1, E).
__device__ __forceinline__ void load_chunk(const int32_t *__restrict__ idx, int c0, int c1,
                                           int E, int (&ev)[kRounds], unsigned &bad) {
    const int lane = threadIdx.x & 31;
    bad = 0;
#pragma unroll
    for (int r = 0; r < kRounds; ++r) {
        const int i = c0 + r * 32 + lane;
        ev[r] = i < c1 ? __ldg(idx + i) : -1;
    }
#pragma unroll
    for (int r = 0; r < kRounds; ++r) {
        if (ev[r] < -1 || ev[r] >= E) {
            bad |= 1u << r;
            ev[r] = -1;
        }
    }
}

__global__ void __launch_bounds__(kThreads)
    tile_hist_kernel(const int32_t *__restrict__ idx, int TK, int E, int tile,
                     int32_t *__restrict__ ws, int32_t *__restrict__ status) {
    extern __shared__ int32_t hist[];  // [E]
    for (int e = threadIdx.x; e < E; e += kThreads) hist[e] = 0;
    __syncthreads();
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int start = blockIdx.x * tile;
    const int end = min(TK, start + tile);
    const int chunk = tile / kWarps;
    const int c0 = start + warp * chunk;
    const int c1 = min(end, c0 + chunk);
    int ev[kRounds];
    unsigned bad;
    load_chunk(idx, c0, c1, E, ev, bad);
#pragma unroll
    for (int r = 0; r < kRounds; ++r) {
        if (c0 + r * 32 >= c1) break;  // warp-uniform
        const unsigned peers = __match_any_sync(kFullMask, ev[r]);
        if (ev[r] >= 0 && lane == __ffs(peers) - 1) atomicAdd(&hist[ev[r]], __popc(peers));
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
    int32_t *wh = sm;                  // [kWarps][E]: per-warp counts, then slot bases
    int32_t *tot = wh + kWarps * E;    // [E] expert histogram
    int32_t *off = tot + E;            // [E+1] first row of each expert
    __shared__ int32_t scan_tmp[kWarps];

    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const bool assigns = blockIdx.x < a.tiles;
    const int tile_id = assigns ? blockIdx.x : 0;
    const int start = tile_id * a.tile;
    const int end = min(a.TK, start + a.tile);
    const int chunk = a.tile / kWarps;
    const int c0 = start + warp * chunk;
    const int c1 = min(end, c0 + chunk);
    const bool need_hist = assigns || a.tiles == 1;

    // With one tile this is the only layout kernel: reset the status word
    // before any error of this CTA is raised (ordered by the barrier below).
    if (a.tiles == 1 && blockIdx.x == 0 && threadIdx.x == 0) *a.status = EP_OK;
    for (int j = threadIdx.x; j < kWarps * E; j += kThreads) wh[j] = 0;

    int ev[kRounds];
    unsigned bad = 0;
    if (need_hist) load_chunk(a.idx, c0, c1, E, ev, bad);
    __syncthreads();

    // 1. per-warp expert histogram of this tile
    if (need_hist) {
#pragma unroll
        for (int r = 0; r < kRounds; ++r) {
            if (c0 + r * 32 >= c1) break;
            const unsigned peers = __match_any_sync(kFullMask, ev[r]);
            if (ev[r] >= 0 && lane == __ffs(peers) - 1) wh[warp * E + ev[r]] += __popc(peers);
            __syncwarp();
        }
    }
    __syncthreads();

    // 2. expert totals; per-warp counts -> per-warp starting slots
    for (int e = threadIdx.x; e < E; e += kThreads) {
        int total = 0, base = 0;
        if (a.tiles == 1) {
            for (int w = 0; w < kWarps; ++w) total += wh[w * E + e];
        } else {
            for (int b = 0; b < a.tiles; ++b) {
                const int c = __ldcg(a.ws + (size_t)b * E + e);
                base += b < tile_id ? c : 0;
                total += c;
            }
        }
        tot[e] = total;
        if (assigns) {
            int run = base;
            for (int w = 0; w < kWarps; ++w) {
                const int c = wh[w * E + e];
                wh[w * E + e] = run;
                run += c;
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
#pragma unroll
        for (int r = 0; r < kRounds; ++r) {
            const int i0 = c0 + r * 32;
            if (i0 >= c1) break;
            const int e = ev[r];
            const unsigned peers = __match_any_sync(kFullMask, e);
            const int slot = e >= 0 ? wh[warp * E + e] + __popc(peers & lanemask_lt()) : 0;
            __syncwarp();
            if (e >= 0 && lane == __ffs(peers) - 1) wh[warp * E + e] += __popc(peers);
            __syncwarp();
            const int i = i0 + lane;
            if (i < c1) {
                int dst = -1;
                if (bad & (1u << r)) {
                    raise_status(a.status, EP_ERR_BAD_EXPERT_ID);
                } else if (e >= 0) {
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
    if (TK <= kMaxTile) {
        p.tiles = 1;
        p.tile = (int)((TK + 511) / 512 * 512);
        if (p.tile == 0) p.tile = 512;
    } else {
        p.tiles = (int)((TK + kMaxTile - 1) / kMaxTile);
        long long per = (TK + p.tiles - 1) / p.tiles;
        p.tile = (int)((per + 511) / 512 * 512);
        p.tiles = (int)((TK + p.tile - 1) / p.tile);
    }
    const bool fill = L.kind == EP_LAYOUT_MASKED && L.row_src != nullptr;
    p.grid = p.tiles;
    if (fill) p.grid = p.tiles > kFillCtas ? p.tiles : (L.num_experts < kFillCtas ? L.num_experts : kFillCtas);
    if (p.grid < p.tiles) p.grid = p.tiles;
    p.smem = sizeof(int32_t) * ((size_t)kWarps * L.num_experts + 2 * (size_t)L.num_experts + 1);
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
