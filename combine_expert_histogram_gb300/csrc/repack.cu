// ep_masked_repack kernel: copy a contiguous layout's expert segments into the
// masked decode slab [E, cap, H] (the "masked-slab repack kernels" of SGLang
// PR "[Feature] Add DeepEPv2 (ElasticBuffer) MoE A2A backend", section
// "Implementation", for both fp32 and packed UE8M0 scales).
//
// Byte copy, HBM-bound.  Every CTA scans m_e = min(count[e], cap) into shared
// memory, then its warps walk the flat list of valid rows grid-stride; a
// binary search over the prefix finds (expert, slot) of a flat row.  One warp
// copies one row: up to 8 KB of it (16 16-byte vectors per lane) and its scale
// words are loaded before any of them is stored, so a row of the DeepSeek-V3
// shape (7168 E4M3 bytes + 56 scale bytes) takes one memory round trip.  The
// loads take the coherent path: non-coherent ones could be moved below the
// stores by the assembler, one vector in flight per lane at a time.
#include "ep_common.cuh"

namespace ep {
namespace {

constexpr int kThreads = 256;
constexpr int kVec = 16;  // 16-byte vectors per lane in flight (8 KB per warp)

__global__ void __launch_bounds__(kThreads)
    repack_kernel(const uint8_t *__restrict__ rows, const uint8_t *__restrict__ row_scales,
                  int row_bytes, int scale_bytes, const int32_t *__restrict__ offset,
                  const int32_t *__restrict__ count, int E, int cap,
                  uint8_t *__restrict__ slab, uint8_t *__restrict__ slab_scales,
                  int32_t *__restrict__ masked_m, int32_t *__restrict__ status,
                  int mn_src_stride, int mn_dst_stride) {
    // mn_src_stride > 0: scale words are MN-major (source column stride over the
    // contiguous row space; destination [E][words][mn_dst_stride])
    extern __shared__ int32_t pre[];  // [E+1]
    __shared__ int32_t scan_tmp[kThreads / 32];
    block_exclusive_scan<kThreads>(
        E, [&](int e) { return min(__ldg(count + e), cap); }, pre, scan_tmp);

    if (blockIdx.x == 0) {
        for (int e = threadIdx.x; e < E; e += kThreads) {
            const int c = __ldg(count + e);
            masked_m[e] = min(c, cap);
            if (c > cap) raise_status(status, EP_ERR_CAPACITY);
        }
    }

    const int lane = threadIdx.x & 31;
    const int total = pre[E];
    const int warps = gridDim.x * (kThreads / 32);
    const int words = scale_bytes / 4;
    const uint32_t *ss_all = reinterpret_cast<const uint32_t *>(row_scales);
    uint32_t *ds_all = reinterpret_cast<uint32_t *>(slab_scales);
    for (int r = blockIdx.x * (kThreads / 32) + (threadIdx.x >> 5); r < total; r += warps) {
        int lo = 0, hi = E;  // pre[lo] <= r < pre[hi]
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (pre[mid] <= r) lo = mid; else hi = mid;
        }
        const int s = r - pre[lo];
        const size_t src = (size_t)__ldg(offset + lo) + s;
        const size_t dst = (size_t)lo * cap + s;
        const uint8_t *sp = rows + src * row_bytes;
        uint8_t *dp = slab + dst * row_bytes;
        // the first scale word of each lane travels with the first part of the row
        uint32_t sw = 0;
        if (lane < words)
            sw = (uint32_t)ld_dep(reinterpret_cast<const int32_t *>(
                mn_src_stride ? ss_all + (size_t)lane * mn_src_stride + src
                              : ss_all + src * words + lane));
        for (int b0 = 0; b0 < row_bytes; b0 += kVec * 32 * 16) {
            uint4 v[kVec];
#pragma unroll
            for (int u = 0; u < kVec; ++u) {
                const int b = b0 + (u * 32 + lane) * 16;
                v[u] = b < row_bytes ? ld_stream_coh(sp + b) : make_uint4(0, 0, 0, 0);
            }
#pragma unroll
            for (int u = 0; u < kVec; ++u) {
                const int b = b0 + (u * 32 + lane) * 16;
                if (b < row_bytes) st_v4(dp + b, v[u]);
            }
        }
        if (lane < words) {
            if (mn_src_stride)
                ds_all[((size_t)lo * words + lane) * mn_dst_stride + s] = sw;
            else
                ds_all[dst * words + lane] = sw;
        }
        for (int b = lane + 32; b < words; b += 32) {  // rows of more than 32 scale words
            if (mn_src_stride)
                ds_all[((size_t)lo * words + b) * mn_dst_stride + s] =
                    __ldg(ss_all + (size_t)b * mn_src_stride + src);
            else
                ds_all[dst * words + b] = __ldg(ss_all + src * words + b);
        }
    }
}

}  // namespace

cudaError_t launch_masked_repack(const ep_layout_t &L, const void *rows,
                                 const void *row_scales, int H, ep_quant_t quant, int cap,
                                 void *slab, void *slab_scales, int32_t *masked_m,
                                 cudaStream_t stream) {
    const int E = L.num_experts;
    const int row_bytes = quant == EP_QUANT_NONE ? 2 * H : H;
    const int G = H / 128;
    const int scale_bytes = (quant == EP_QUANT_FP8_F32 || quant == EP_QUANT_MXFP8) ? 4 * G
                            : (quant == EP_QUANT_FP8_UE8M0 || quant == EP_QUANT_FP8_UE8M0_MN)
                                ? 4 * ((G + 3) / 4) : 0;
    int mn_src = 0, mn_dst = 0;
    if (quant == EP_QUANT_FP8_UE8M0_MN) {
        const long long TK = (long long)L.num_tokens * L.num_topk;
        const long long rows_cap = TK + (TK < E ? TK : E) * (long long)(L.align - 1);
        mn_src = (int)((rows_cap + 3) / 4 * 4);
        mn_dst = (cap + 3) / 4 * 4;
    }
    // Enough warps to keep HBM busy (with a row of up to 8 KB in flight per
    // warp, 16 warps per SM hold ~18 MB); the valid rows number at most T*K.
    const long long rows_max = (long long)L.num_tokens * L.num_topk;
    long long blocks = (rows_max + kThreads / 32 - 1) / (kThreads / 32);
    const long long limit = 2LL * sm_count();
    if (blocks > limit) blocks = limit;
    if (blocks < 1) blocks = 1;
    const size_t smem = sizeof(int32_t) * (size_t)(E + 1);
    repack_kernel<<<(unsigned)blocks, kThreads, smem, stream>>>(
        static_cast<const uint8_t *>(rows), static_cast<const uint8_t *>(row_scales), row_bytes,
        scale_bytes, L.expert_offset, L.expert_count, E, cap, static_cast<uint8_t *>(slab),
        static_cast<uint8_t *>(slab_scales), masked_m, L.status, mn_src, mn_dst);
    return cudaGetLastError();
}

}  // namespace ep
