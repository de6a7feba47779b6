// The decode-sized layout (up to kClusterMaxEntries top-k entries) computed
// by thread-block clusters in one kernel: one cluster ranks the entries, 1-3
// more only count them.  The device body of the layout kernel in
// csrc/layout.cu, and its host-side sizing and launch.
//
// The layout step that DeepEP V2's dispatch performs internally ("infers the
// layout from topk_idx", SGLang PR "moe: add DeepEP V2 ElasticBuffer support
// to MoE token dispatcher", section "Motivation"), for the contiguous
// (prefill) and masked (decode) layouts of SGLang PR "[Feature] Add DeepEPv2
// (ElasticBuffer) MoE A2A backend", section "Supported scope".
#pragma once

#include "ep_common.cuh"

namespace ep {
namespace cl {

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
__device__ __forceinline__ void cluster_arrive_relaxed() {
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Shared-memory address `a` of this CTA, as the same address in the CTA of
// cluster rank `rank` (distributed shared memory).
__device__ __forceinline__ uint32_t peer_addr(uint32_t a, unsigned rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(rank));
    return r;
}
// Bulk copy of `bytes` (a multiple of 16, both addresses 16-byte aligned)
// from this CTA's shared memory at `src` to address `dst` of a peer CTA,
// counted against the transaction bytes of the peer's barrier `bar` (both
// already mapped to the peer).
__device__ __forceinline__ void push_to_peer(uint32_t dst, uint32_t src, uint32_t bytes,
                                             uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        ::"r"(dst), "r"(src), "r"(bytes), "r"(bar)
        : "memory");
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

__host__ __device__ inline int round_up_pow2(int v, int a) { return (v + a - 1) & ~(a - 1); }

// Grid: one or more clusters.  Every cluster splits the TK entries the same
// way (CTA c of a cluster owns entries [c * 8 * chunk, (c + 1) * 8 * chunk),
// warp w of it the chunk at w * chunk), so (CTA, warp, round, lane) order is
// entry order and the slot of an entry is
//   (entries of its expert in lower CTAs) + (in lower warps of its CTA)
//   + (in earlier rounds of its warp) + (in lower lanes of its round).
// Cluster 0 (RANK) ranks the entries and writes dst_row and the valid
// row_src rows; the 1-3 clusters after it only count (shared-memory atomics)
// and write the counts, offsets, status word and rank rows (cluster 1) and
// the -1 rows of row_src (all of them).  So the fill runs on more SMs and in
// parallel with the slot writes (Qwen3-30B-A3B decode 3.02 -> 2.73 us,
// DeepSeek-V3 decode 4.23 -> 3.74 us against two clusters that both ranked
// and shared the fill).
//
// The CTAs exchange their histograms by pushing: each CTA bulk-copies its
// histogram block into a slot of every peer's shared memory, and the copies
// complete on the peer's barrier, so every CTA waits for its own incoming
// bytes only.  Measured against pulling the peers' words with
// distributed-shared-memory loads after a cluster barrier (4-byte or 16-byte
// loads, four peers at a time) and against 16-byte remote stores followed by
// a cluster barrier: 0.4-0.5 us faster at 8 CTAs and 2048 entries, 0.4-0.75
// us faster at 16 CTAs and 8192 entries.
//
// The body of a layout kernel of kClThreads threads per CTA: `csm` is
// cluster_smem(E) bytes of the CTA's dynamic shared memory (16-byte
// aligned).  The caller has waited for the previous kernel on the stream
// (griddepcontrol.wait) before calling it; every thread of every CTA of the
// grid calls it.  Ends with a cluster barrier.
template <int ROUNDS, bool RANK>
__device__ __forceinline__ void cluster_layout_body(const ClusterArgs &a, int32_t *csm) {
    const int E = a.E;
    const int E4 = round_up_pow2(E, 4);  // whole 16-byte words of counts
    const int HW = E4 + 4;               // words of a histogram block: counts, flag word, padding
    int32_t *wh = csm;                   // [kClWarps][E] per-warp counts, then warp bases
    int32_t *hist = wh + kClWarps * E;   // [HW] this CTA's block: counts (0 past E), [E4] bad-id flag
    int32_t *tot = hist + HW;            // [E4] expert totals
    int32_t *base = tot + E4;            // [E4] entries of each expert in lower CTAs
    int32_t *off = base + E4;            // [E4 + 4] first row of each expert (E + 1 used)
    int32_t *recv = off + E4 + 4;        // [kClMaxCtas][HW] the peers' blocks, by cluster rank
    __shared__ int32_t scan_tmp[kClWarps];
    __shared__ int32_t s_flags;  // bit 0: a bad id; 1: a masked expert over capacity; 2: timeout
    __shared__ __align__(8) uint64_t s_bar;  // completes when every peer's block has arrived

    const unsigned crank = cluster_ctarank(), csize = cluster_nctarank();
    constexpr bool writer = RANK, meta = !RANK;
    const bool meta_writer = meta && blockIdx.x / csize == 1;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int w0 = ((int)crank * kClWarps + warp) * a.chunk;
    const int w1 = min(a.TK, w0 + a.chunk);
    if (threadIdx.x == 0) {
        mbar_init(&s_bar, 1);
        mbar_init_fence();
    }
    // the barrier is initialised before any peer may push (the matching
    // wait comes after the ranking, so this costs nothing)
    cluster_arrive_relaxed();

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
    if constexpr (!RANK) {  // counts only
#pragma unroll
        for (int r = 0; r < ROUNDS; ++r) {
            const int e0 = ev[r];
            bad |= e0 < -1 || e0 >= E;
            if (e0 >= 0 && e0 < E) atomicAdd(&row[e0], 1);
        }
    } else {
#pragma unroll
    for (int r = 0; r < ROUNDS; ++r) {
        const int e0 = ev[r];
        bad |= e0 < -1 || e0 >= E;
        const int e = (e0 >= 0 && e0 < E) ? e0 : E;  // E = no expert
        ev[r] = e;
        // lanes with the same expert: one ballot per bit of the id (E itself
        // must fit); the ballots are independent, so their latencies overlap.
        // In this latency-bound kernel (about one round per warp) they
        // measured 0.2-0.35 us faster than one __match_any_sync, whose single
        // result comes later; the tiled kernel's many rounds prefer the latter.
        unsigned peers = kFullMask;
        const int nbits = 32 - __clz(E);
        for (int b = 0; b < nbits; ++b) {
            const unsigned bit = (e >> b) & 1u;
            const unsigned bal = __ballot_sync(kFullMask, bit);
            peers &= bit ? bal : ~bal;
        }
        const int before = e < E ? row[e] : 0;
        __syncwarp();
        if (e < E && lane == __ffs(peers) - 1) row[e] = before + __popc(peers);
        __syncwarp();
        rank[r] = before + __popc(peers & lanemask_lt());
    }
    }
    bad = __syncthreads_or(bad);

    // 3. warp counts -> warp bases within the CTA; the CTA's histogram block
    for (int e = threadIdx.x; e < E4; e += kClThreads) {
        int run = 0;
        if (e < E) {
#pragma unroll
            for (int w = 0; w < kClWarps; ++w) {
                const int c = wh[w * E + e];
                wh[w * E + e] = run;
                run += c;
            }
        }
        hist[e] = run;
    }
    if (threadIdx.x < 4) hist[E4 + threadIdx.x] = threadIdx.x == 0 ? bad : 0;
    fence_proxy_async_smem();  // the block is read by the bulk copies below
    __syncthreads();

    // 4. push the block into slot crank of every peer; wait for the peers'
    //    blocks; totals, this CTA's base and the error flags from them
    cluster_wait();  // every peer's barrier is initialised
    // lane 0 of warp w copies to peers w, w + 8: spreading the copies over
    // the warps measured 0.2-0.4 us faster than one thread issuing all of
    // them (and than the lanes of one warp issuing one each)
    if (lane == 0) {
        const uint32_t bytes = (uint32_t)HW * sizeof(int32_t);
        const uint32_t bar = smem_addr(&s_bar);
        if (warp == 0)
            asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar),
                         "r"(bytes * (csize - 1))
                         : "memory");
        const uint32_t src = smem_addr(hist), dst = smem_addr(recv + crank * HW);
        for (unsigned p = warp; p < csize; p += kClWarps)
            if (p != crank) push_to_peer(peer_addr(dst, p), src, bytes, peer_addr(bar, p));
    }
    int flags = mbar_wait(&s_bar, 0, nullptr) ? 0 : 4;
    const int cap = a.cap, masked = a.masked;
    for (int e = threadIdx.x; e < E; e += kClThreads) {
        int t = 0, b = 0;
        for (unsigned c = 0; c < csize; ++c) {
            const int v = c == crank ? hist[e] : recv[c * HW + e];
            t += v;
            b += c < crank ? v : 0;
        }
        tot[e] = t;
        base[e] = b;
        if (masked && t > cap) flags |= 2;
    }
    if (threadIdx.x < csize && (threadIdx.x == crank ? hist[E4] : recv[threadIdx.x * HW + E4]))
        flags |= 1;
    // every copy into this CTA has landed (nothing to publish: relaxed); the
    // peers may exit once every thread of the cluster has arrived here, as
    // then no copy still reads their shared memory
    cluster_arrive_relaxed();
    if (flags) atomicOr(&s_flags, flags);
    // A timed-out wait (a bulk copy that never completed) reaches the status
    // word from CTA 0 of cluster 1 through its flags, and from any other CTA
    // as a raise: that comes a second after the exchange began, long after
    // that CTA (which finished its own exchange, or it would report the
    // timeout itself) wrote the word.
    if (flags & 4) raise_status(a.status, EP_ERR_TIMEOUT);

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
                    // slot < tot[e] always holds unless the exchange timed out
                    // (then the counts are garbage): no row outside the expert's
                    if (slot < tot[e] && !(masked && slot >= cap)) dst = off[e] + slot;
                }
                a.dst_row[i] = dst;
                if (dst >= 0 && a.row_src) a.row_src[dst] = i;
            }
        }
    }
    if (meta_writer) {
        // 7. counts and offsets, a slice of the experts per CTA; the status
        //    word from CTA 0, the rank rows from the last CTA
        for (int e = (int)crank * kClThreads + threadIdx.x; e < E; e += (int)csize * kClThreads) {
            a.count[e] = tot[e];
            a.offset[e] = off[e];
        }
        if (crank == 0 && threadIdx.x == 0) {
            const int f = s_flags;
            *a.status = (f & 4)   ? EP_ERR_TIMEOUT
                        : (f & 1) ? EP_ERR_BAD_EXPERT_ID
                        : (f & 2) ? EP_ERR_CAPACITY
                                  : EP_OK;
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
    //    one warp per expert across the counting clusters
    if (a.row_src && meta) {
        const int gw = ((int)blockIdx.x - (int)csize) * kClWarps + warp;
        const int nw = ((int)gridDim.x - (int)csize) * kClWarps;
        for (int e = gw; e < E; e += nw) {
            const int r0 = off[e] + (masked ? min(tot[e], cap) : tot[e]);
            const int r1 = masked ? off[e] + cap : off[e + 1];
            fill_minus_one(a.row_src, r0, r1, lane);
        }
    }
    // no CTA leaves while a copy may still read its shared memory
    cluster_wait();
}

// Dynamic shared memory of the layout body: per-warp counts, the CTA's
// histogram block, totals, bases, offsets and one block per possible peer.
inline size_t cluster_smem(int E) {
    const size_t E4 = (size_t)round_up_pow2(E, 4), HW = E4 + 4;
    return sizeof(int32_t) * ((size_t)kClWarps * E + HW + 2 * E4 + (E4 + 4) + kClMaxCtas * HW);
}

// CTAs of one cluster for TK entries with at most max_ctas per cluster, and
// the entries per warp (32 x a power-of-two number of rounds).
inline void cluster_shape(long long TK, int max_ctas, int *ctas, int *chunk) {
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

constexpr int kFillRowsPerCta = 2048;  // row_src rows a filling CTA is given, at most
constexpr int kMaxMetaClusters = 3;

// Clusters of the launch: the ranking cluster plus 1-3 counting clusters for
// the counts, offsets, status and rank rows and the row_src fill, enough to
// give each of their CTAs about kFillRowsPerCta rows of the largest possible
// fill (E x capacity masked, E x (align - 1) padding rows contiguous; one
// without row_src).  The fill is bound by each SM's store rate (about 30
// bytes per clock), so it wants SMs; off the ranking cluster neither it nor
// the metadata stores delay the slot writes (without row_src one counting
// cluster measured 0.3 us faster than one cluster doing everything).
inline int fill_clusters(const ep_layout_t &L, int ctas) {
    if (L.row_src == nullptr) return 2;
    const long long rows = L.kind == EP_LAYOUT_MASKED
                               ? (long long)L.num_experts * L.capacity
                               : (long long)L.num_experts * (L.align - 1);
    const long long per = (long long)ctas * kFillRowsPerCta;
    long long m = (rows + per - 1) / per;
    if (m < 1) m = 1;
    if (m > kMaxMetaClusters) m = kMaxMetaClusters;
    return 1 + (int)m;
}

// The layout body's arguments for layout L.
inline ClusterArgs cluster_args(const int32_t *topk_idx, const ep_layout_t &L, int chunk) {
    ClusterArgs c;
    c.idx = topk_idx;
    c.TK = L.num_tokens * L.num_topk;
    c.E = L.num_experts;
    c.R = L.num_ranks;
    c.masked = L.kind == EP_LAYOUT_MASKED;
    c.align = c.masked ? 1 : L.align;
    c.cap = c.masked ? L.capacity : 0;
    c.chunk = chunk;
    c.dst_row = L.dst_row;
    c.row_src = L.row_src;
    c.count = L.expert_count;
    c.offset = L.expert_offset;
    c.rank_rows = L.rank_rows;
    c.status = L.status;
    return c;
}

// Largest cluster (16 CTAs, else the portable 8) that the device can
// co-schedule for kernel `func` of kClThreads threads and `smem` bytes of
// dynamic shared memory; once per device and kernel.  Sets the kernel's
// dynamic shared-memory limit and non-portable-cluster attribute.
int max_cluster_ctas(const void *func, size_t smem);

// Launch `func(args...)` as `clusters` clusters of `ctas` CTAs of kClThreads
// threads, optionally as a programmatic dependent of the previous kernel.
template <typename... KArgs, typename... Args>
cudaError_t launch_clusters(void (*func)(KArgs...), int ctas, int clusters, size_t smem,
                            cudaStream_t stream, bool programmatic, Args... args) {
    cudaError_t err = allow_dynamic_smem(func, smem);
    if (err != cudaSuccess) return err;
    if (ctas > 8) {
        err = cudaFuncSetAttribute(func, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        if (err != cudaSuccess) return err;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(ctas * clusters);
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
    cfg.numAttrs = programmatic ? 2 : 1;
    return cudaLaunchKernelEx(&cfg, func, static_cast<KArgs>(args)...);
}

}  // namespace cl
}  // namespace ep
