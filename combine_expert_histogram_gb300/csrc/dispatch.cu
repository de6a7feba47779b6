// ep_dispatch kernels: scatter token rows into the layout, fused with dynamic
// 1x128 FP8-E4M3 quantisation (fp32 or packed UE8M0 scales) or 1x32 MXFP8.
//
// Format and scale conventions follow SGLang PR "[Feature] Add DeepEPv2
// (ElasticBuffer) MoE A2A backend" ("Supported scope": dynamic blockwise FP8;
// "Implementation": Hopper FP32 scales and Blackwell packed UE8M0 scales) and
// the vLLM tools/ep_kernels deepep_v2 commit ("FP8 block-quantized dispatch");
// MXFP8 is the "1x32 MXFP8 ... with dynamic activation scaling" format of the
// SGLang discussion "deepep v2 support?", scaled by the OCP Microscaling (MX)
// v1.0 rule X = 2^(floor(log2 amax) - 8).
//
// HBM-bound: each token row is read once and written K times (80 % of the
// bytes are writes).  Persistent CTAs take tokens c, c + gridDim.x, ...; the
// rows move through shared memory by TMA bulk copies:
//   - a producer warp keeps a ring of `stages` x rows in flight (one
//     cp.async.bulk global -> shared copy per row, completing on the stage's
//     mbarrier), and hands every finished output row to the TMA engine with
//     one bulk store per destination;
//   - FP8: consumer warps take 16 consecutive elements per lane from the x
//     stage (8 lanes per 1x128 group, amax by three xor-shuffles), write the
//     E4M3 bytes into one of kOutBufs output rows and store the scale words
//     directly from registers (gathered by shuffles); full / empty mbarrier
//     pairs pass x stages and output rows between the two roles, so the
//     quantisation of one token overlaps the bulk stores of the ones before;
//   - bf16 rows need no conversion: one warp stores them straight from the
//     x stage.
// With few tokens per SM (decode) the ring only adds latency: there each warp
// owns 32 slots of a row in registers and stores its 16 bytes per lane to the
// K destinations itself (no shared memory, no barriers), the next token's
// slots and destinations in flight meanwhile.
// Dispatch is launched as the layout's programmatic dependent: the first rows
// load while the layout finishes, and destinations are read only after
// griddepcontrol.wait.  Every mbarrier wait is bounded (about a second); on
// expiry the kernel raises EP_ERR_TIMEOUT, waits for the row copies it issued
// to land and returns.  That drain is bounded as well (about a second in
// all): a copy from ordinary global memory lands long before, but if the
// drain itself ran out the CTA would exit with a copy into its shared memory
// still pending, which is undefined; EP_ERR_TIMEOUT is then the only thing the
// kernel guarantees, and the caller should treat the context as suspect.
#include <cuda_fp8.h>

#include "ep_common.cuh"

namespace ep {
namespace {

constexpr int kMaxConsumerWarps = 16;
constexpr int kMaxStages = 8;
constexpr int kStageBudget = 144 * 1024;  // shared memory per CTA aimed for
constexpr int kOutBufs = 4;               // FP8 output rows per CTA, at most
constexpr int kSmemMax = 227 * 1024;      // dynamic shared memory per CTA
constexpr int kCopyMaxStages = 8;         // bf16 rows in flight per CTA, at most
constexpr int kCopyBudget = 144 * 1024;   // bf16: shared memory per CTA aimed for

__device__ __forceinline__ uint32_t fp8x4(float a, float b, float c, float d) {
    // __nv_cvt_float2_to_fp8x2: round to nearest even, saturate to +-448;
    // the first element of the pair lands in the low byte.
    const uint32_t lo = __nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
    const uint32_t hi = __nv_cvt_float2_to_fp8x2(make_float2(c, d), __NV_SATFINITE, __NV_E4M3);
    return (lo & 0xffffu) | (hi << 16);
}

// Bulk copy of `bytes` (multiple of 16, both addresses 16-byte aligned) from
// shared memory to global memory, tracked by the issuing thread's bulk group.
// The destination rows are written once and not read again by this kernel, so
// their L2 lines are marked evict-first (at the DeepSeek-V3 prefill shape this
// measured 1-2 us faster; the same hint on the x loads made the step slower).
__device__ __forceinline__ void bulk_store(void *gdst, const void *ssrc, uint32_t bytes) {
    uint64_t policy;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(policy));
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group.L2::cache_hint [%0], [%1], %2, %3;"
                 ::"l"(gdst), "r"(smem_addr(ssrc)), "r"(bytes), "l"(policy)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Wait until at most N of this thread's bulk groups are still reading their source.
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
    asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}
// Start the row copy global -> shared: arrive on the barrier, announcing
// `bytes` of transactions, and issue one bulk copy that completes them.
__device__ __forceinline__ void load_row(void *sdst, const void *gsrc, uint32_t bytes,
                                         uint64_t *bar) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
                 "r"(bytes)
                 : "memory");
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
            "r"(smem_addr(sdst)),
        "l"(gsrc), "r"(bytes), "r"(smem_addr(bar))
        : "memory");
}

// Quantise one FP8 slot (16 consecutive elements a, b of group j/8, part
// lane%8 of its 8 lanes).  Returns the 16 E4M3 bytes; `sc` receives the
// group's fp32 scale bits (FP8_F32), its UE8M0 exponent byte (FP8_UE8M0*), or
// the E8M0 byte of the slot's 32-element block (MXFP8, shared by a lane pair).
// Every lane of the warp must call it (shuffles over the whole warp).
template <int Q>
__device__ __forceinline__ uint4 quant_slot(uint4 a, uint4 b, int lane, uint32_t &sc) {
    const unsigned gmask = 0xffu << (lane & 24);
    float v[16];
    const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        v[2 * i] = bf16_lo(w[i]);
        v[2 * i + 1] = bf16_hi(w[i]);
    }
    uint4 q;
    if (Q == EP_QUANT_MXFP8) {
        // two lanes hold one 32-element block: X = 2^(floor(log2 amax) - 8),
        // clamped at 2^-127; byte = log2(X) + 127; multiply by 1/X = 2^(127-byte)
        float bmax = 0.0f;
#pragma unroll
        for (int i = 0; i < 16; ++i) bmax = fmaxf(bmax, fabsf(v[i]));
        bmax = fmaxf(bmax, __shfl_xor_sync(gmask, bmax, 1));
        const int be = (int)((__float_as_uint(bmax) >> 23) & 0xffu);  // 0: zero/subnormal
        const int byte = be > 8 ? be - 8 : 0;
        const float inv = __uint_as_float((uint32_t)(254 - byte) << 23);
        q.x = fp8x4(__fmul_rn(v[0], inv), __fmul_rn(v[1], inv), __fmul_rn(v[2], inv), __fmul_rn(v[3], inv));
        q.y = fp8x4(__fmul_rn(v[4], inv), __fmul_rn(v[5], inv), __fmul_rn(v[6], inv), __fmul_rn(v[7], inv));
        q.z = fp8x4(__fmul_rn(v[8], inv), __fmul_rn(v[9], inv), __fmul_rn(v[10], inv), __fmul_rn(v[11], inv));
        q.w = fp8x4(__fmul_rn(v[12], inv), __fmul_rn(v[13], inv), __fmul_rn(v[14], inv), __fmul_rn(v[15], inv));
        sc = (uint32_t)byte;
    } else {
        float amax = 0.0f;
#pragma unroll
        for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(v[i]));
        amax = fmaxf(amax, __shfl_xor_sync(gmask, amax, 4));
        amax = fmaxf(amax, __shfl_xor_sync(gmask, amax, 2));
        amax = fmaxf(amax, __shfl_xor_sync(gmask, amax, 1));
        // s = max(amax, 1e-4) / 448, an IEEE round-to-nearest division.
        const float s = __fdiv_rn(fmaxf(amax, 1e-4f), 448.0f);
        if (Q == EP_QUANT_FP8_F32) {
            q.x = fp8x4(__fdiv_rn(v[0], s), __fdiv_rn(v[1], s), __fdiv_rn(v[2], s), __fdiv_rn(v[3], s));
            q.y = fp8x4(__fdiv_rn(v[4], s), __fdiv_rn(v[5], s), __fdiv_rn(v[6], s), __fdiv_rn(v[7], s));
            q.z = fp8x4(__fdiv_rn(v[8], s), __fdiv_rn(v[9], s), __fdiv_rn(v[10], s), __fdiv_rn(v[11], s));
            q.w = fp8x4(__fdiv_rn(v[12], s), __fdiv_rn(v[13], s), __fdiv_rn(v[14], s), __fdiv_rn(v[15], s));
            sc = __float_as_uint(s);
        } else {
            // scale rounded up to a power of two 2^(e-127); multiply by 2^(127-e)
            const uint32_t bits = __float_as_uint(s);
            const int e = (int)((bits >> 23) & 0xffu) + ((bits & 0x7fffffu) != 0u);
            const float inv = __uint_as_float((uint32_t)(254 - e) << 23);
            q.x = fp8x4(__fmul_rn(v[0], inv), __fmul_rn(v[1], inv), __fmul_rn(v[2], inv), __fmul_rn(v[3], inv));
            q.y = fp8x4(__fmul_rn(v[4], inv), __fmul_rn(v[5], inv), __fmul_rn(v[6], inv), __fmul_rn(v[7], inv));
            q.z = fp8x4(__fmul_rn(v[8], inv), __fmul_rn(v[9], inv), __fmul_rn(v[10], inv), __fmul_rn(v[11], inv));
            q.w = fp8x4(__fmul_rn(v[12], inv), __fmul_rn(v[13], inv), __fmul_rn(v[14], inv), __fmul_rn(v[15], inv));
            sc = (uint32_t)e;
        }
    }
    return q;
}

// Scale words of one warp pass (first slot wbase = j - lane) for every
// destination: lanes k < K hold destination k in `cd`; `sc` as quant_slot
// returned it; G groups, `words` scale words per row.
template <int Q>
__device__ __forceinline__ void store_scales(uint32_t *scales, uint32_t sc, int j, int lane,
                                             int slots, int cd, int K, int G, int words,
                                             int mn_stride, int mn_cap) {
    const int wbase = j - lane;
    if constexpr (Q == EP_QUANT_FP8_F32) {
        // group j/8's scale: lane sub of the group writes it for k = sub, sub+8, ...
        for (int kb = 0; kb < K; kb += 8) {
            const int k = kb + (lane & 7);
            const int d = __shfl_sync(kFullMask, cd, k & 31);
            if (j < slots && k < K && d >= 0) scales[(size_t)d * G + (j >> 3)] = sc;
        }
    } else if constexpr (Q == EP_QUANT_MXFP8) {
        // the warp's 16 blocks make 4 words (word wi: slots 8wi .. 8wi+7, one
        // byte per lane pair); lane 8wi + k%8 writes word wi for k
        const int wi = lane >> 3;
        uint32_t word = 0;
#pragma unroll
        for (int m = 0; m < 4; ++m) word |= __shfl_sync(kFullMask, sc, 8 * wi + 2 * m) << (8 * m);
        const int g = (wbase >> 3) + wi;  // the word's index in the scale row
        for (int kb = 0; kb < K; kb += 8) {
            const int k = kb + (lane & 7);
            const int d = __shfl_sync(kFullMask, cd, k & 31);
            if (g < G && k < K && d >= 0) scales[(size_t)d * G + g] = word;
        }
    } else {
        // UE8M0: the warp's 4 groups make one word, byte m = group wbase/8 + m
        // (127 = 2^0 past the last group); lane k writes it for destination k
        uint32_t word = 0;
#pragma unroll
        for (int m = 0; m < 4; ++m) {
            const uint32_t e = __shfl_sync(kFullMask, sc, 8 * m);
            word |= ((wbase >> 3) + m < G ? e : 127u) << (8 * m);
        }
        const int wd = wbase >> 5;
        if (lane < K && cd >= 0) {
            size_t at = (size_t)cd * words + wd;
            if (Q == EP_QUANT_FP8_UE8M0_MN)  // word wd of row d at wd*stride + d, per expert if masked
                at = mn_cap ? ((size_t)(cd / mn_cap) * words + wd) * mn_stride + (size_t)(cd % mn_cap)
                            : (size_t)wd * mn_stride + cd;
            scales[at] = word;
        }
    }
}

// Tokens of CTA c in a persistent grid: c, c + step, ...
__device__ __forceinline__ int cta_tokens(int T, int step) {
    return T > (int)blockIdx.x ? (T - 1 - (int)blockIdx.x) / step + 1 : 0;
}

// FP8 dispatch: warp 0 produces (lane 0 drives the TMA), warps 1..C consume.
// Token i of the CTA uses x stage i % stages and output row i % nob.
template <int Q>
__global__ void __launch_bounds__(32 * (kMaxConsumerWarps + 1))
    quant_kernel(const uint16_t *__restrict__ x, int T, int K, int H, const int32_t *dst_row,
                 uint8_t *__restrict__ out, uint32_t *__restrict__ scales, const float *topk_w,
                 float *__restrict__ row_w, int32_t *status, int mn_stride, int mn_cap,
                 int stages, int xstage_bytes, int nob) {
    extern __shared__ __align__(128) uint8_t smem[];  // [stages] x rows, [nob] E4M3 rows
    __shared__ __align__(8) uint64_t xfull[kMaxStages], xempty[kMaxStages];
    __shared__ __align__(8) uint64_t ofull[kOutBufs], oempty[kOutBufs];
    __shared__ int s_loads[kMaxStages];  // rows requested per stage, for the drain
    __shared__ int s_fail;
    constexpr bool kUe8m0 = Q == EP_QUANT_FP8_UE8M0 || Q == EP_QUANT_FP8_UE8M0_MN;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int C = (blockDim.x >> 5) - 1;  // consumer warps
    const int G = H >> 7, slots = G * 8;
    const int words = kUe8m0 ? (G + 3) >> 2 : G;
    const uint32_t x_bytes = 2u * (uint32_t)H;
    const int step = gridDim.x;
    const int n = cta_tokens(T, step);
    uint8_t *orows = smem + (size_t)stages * xstage_bytes;
    const volatile int *fail = &s_fail;
    // the next kernel (combine) waits for this one itself: let it launch now
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    if (threadIdx.x == 0) {
        for (int s = 0; s < stages; ++s) {
            mbar_init(&xfull[s], 1);
            mbar_init(&xempty[s], C);
            s_loads[s] = 0;
        }
        for (int b = 0; b < nob; ++b) {
            mbar_init(&ofull[b], C);
            mbar_init(&oempty[b], 1);
        }
        s_fail = 0;
        mbar_init_fence();
    }
    __syncthreads();

    if (warp == 0) {
        // ---- producer: x rows in, finished rows out ----
        if (lane == 0)
            for (int i = 0; i < stages && i < n; ++i) {
                load_row(smem + (size_t)i * xstage_bytes, x + (size_t)(blockIdx.x + i * step) * H,
                         x_bytes, &xfull[i]);
                s_loads[i] = 1;
            }
        // x was complete before the layout started; dst_row is the layout's
        // output (a no-op without a programmatic edge)
        asm volatile("griddepcontrol.wait;" ::: "memory");
        int cd = n > 0 && lane < K ? ld_dep(dst_row + (size_t)blockIdx.x * K + lane) : -1;
        for (int i = 0; i < n; ++i) {
            const int t = blockIdx.x + i * step;
            const int nd = i + 1 < n && lane < K ? ld_dep(dst_row + (size_t)(t + step) * K + lane) : -1;
            const int b = i % nob;
            const bool ok = mbar_wait(&ofull[b], (i / nob) & 1, fail);
            if (__any_sync(kFullMask, !ok)) {  // the whole warp leaves together
                s_fail = 1;
                break;
            }
            const uint8_t *orow = orows + (size_t)b * H;
            for (int k = 0; k < K; ++k) {
                const int d = __shfl_sync(kFullMask, cd, k);
                if (lane == 0 && d >= 0) bulk_store(out + (size_t)d * H, orow, (uint32_t)H);
            }
            if (lane == 0) {
                bulk_commit();
                if (i > 0) {  // the previous row is free once its stores have read it
                    bulk_wait_read<1>();
                    mbar_arrive(&oempty[(i - 1) % nob]);
                }
            }
            if (i + stages < n) {  // refill this token's x stage once every consumer read it
                const int s = i % stages;
                const bool ok2 = mbar_wait(&xempty[s], (i / stages) & 1, fail);
                if (__any_sync(kFullMask, !ok2)) {
                    s_fail = 1;
                    break;
                }
                if (lane == 0) {
                    load_row(smem + (size_t)s * xstage_bytes, x + (size_t)(t + stages * step) * H,
                             x_bytes, &xfull[s]);
                    ++s_loads[s];
                }
            }
            cd = nd;
        }
        if (lane == 0) bulk_wait_read<0>();  // the rows must outlive the bulk reads
    } else {
        // ---- consumers: quantise x stage -> output row, scales from registers ----
        const int w = warp - 1;
        const bool weights = row_w != nullptr && w == 0 && lane < K;
        const int j0 = w * 32 + lane;
        // x was complete before the layout started: when one pass covers the
        // row, the first token is quantised while the layout may still run
        // and only its scale words wait for the destinations
        bool early = n > 0 && slots <= C * 32;
        uint32_t sc0 = 0;
        if (early) {
            const bool ok = mbar_wait(&xfull[0], 0, fail);  // output row 0 starts free
            if (__any_sync(kFullMask, !ok)) {
                s_fail = 1;
                early = false;
            } else {
                const uint4 *xv = reinterpret_cast<const uint4 *>(smem);
                uint4 a = make_uint4(0, 0, 0, 0), a2 = a;
                if (j0 < slots) {
                    a = xv[2 * j0];
                    a2 = xv[2 * j0 + 1];
                }
                const uint4 q = quant_slot<Q>(a, a2, lane, sc0);
                if (j0 < slots) reinterpret_cast<uint4 *>(orows)[j0] = q;
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(&xempty[0]);
                    mbar_arrive(&ofull[0]);
                }
            }
        }
        asm volatile("griddepcontrol.wait;" ::: "memory");
        int cd = n > 0 && lane < K ? ld_dep(dst_row + (size_t)blockIdx.x * K + lane) : -1;
        float cw = n > 0 && weights ? ld_dep(topk_w + (size_t)blockIdx.x * K + lane) : 0.0f;
        for (int i = 0; i < n && !*fail; ++i) {
            const int t = blockIdx.x + i * step;
            int nd = -1;
            float nw = 0.0f;
            if (i + 1 < n && lane < K) {
                nd = ld_dep(dst_row + (size_t)(t + step) * K + lane);
                if (weights) nw = ld_dep(topk_w + (size_t)(t + step) * K + lane);
            }
            if (i == 0 && early) {  // quantised above: the scale words remain
                store_scales<Q>(scales, sc0, j0, lane, slots, cd, K, G, words, mn_stride, mn_cap);
                if (weights && cd >= 0) row_w[cd] = cw;
                cd = nd;
                cw = nw;
                continue;
            }
            const int s = i % stages, b = i % nob;
            const bool ok = mbar_wait(&xfull[s], (i / stages) & 1, fail) &&
                            mbar_wait(&oempty[b], ((i / nob) & 1) ^ 1, fail);
            if (__any_sync(kFullMask, !ok)) {  // the whole warp leaves together
                s_fail = 1;
                break;
            }
            const uint4 *xv = reinterpret_cast<const uint4 *>(smem + (size_t)s * xstage_bytes);
            uint4 *orow = reinterpret_cast<uint4 *>(orows + (size_t)b * H);
            for (int j = w * 32 + lane; j - lane < slots; j += C * 32) {  // whole warps per pass
                uint4 a = make_uint4(0, 0, 0, 0), a2 = a;
                if (j < slots) {
                    a = xv[2 * j];
                    a2 = xv[2 * j + 1];
                }
                uint32_t sc;
                const uint4 q = quant_slot<Q>(a, a2, lane, sc);
                if (j < slots) orow[j] = q;
                store_scales<Q>(scales, sc, j, lane, slots, cd, K, G, words, mn_stride, mn_cap);
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&xempty[s]);
                mbar_arrive(&ofull[b]);
            }
            if (weights && cd >= 0) row_w[cd] = cw;
            cd = nd;
            cw = nw;
        }
    }
    __syncthreads();
    if (s_fail && threadIdx.x == 0) {
        // every thread passed griddepcontrol.wait, so the status word is ours
        // to raise; let each stage's last row copy land before the shared
        // memory is released
        raise_status(status, EP_ERR_TIMEOUT);
        const long long t0 = clock64();
        for (int s = 0; s < stages; ++s) {
            const long long left = kWaitLimit - (clock64() - t0);
            if (s_loads[s] > 0 && (left <= 0 || !mbar_wait(&xfull[s], (s_loads[s] - 1) & 1, nullptr, left)))
                break;
        }
    }
}

// Slot j of token row xr into registers: 16 bf16 (two 16-byte loads) for the
// FP8 modes, 8 bf16 for bf16.  Coherent loads: the next token's slot is loaded
// ahead of the current token's stores and must stay there (a non-coherent
// load could be moved below them).
template <int Q>
__device__ __forceinline__ void load_slot(const uint16_t *xr, int j, uint4 &a, uint4 &b) {
    if (Q == EP_QUANT_NONE) {
        a = ld_stream_coh(xr + j * 8);
    } else {
        a = ld_stream_coh(xr + j * 16);
        b = ld_stream_coh(xr + j * 16 + 8);
    }
}

// Dispatch token t from registers: thread i owns slots i, i + blockDim.x, ...
// (whole warps step through the passes, lanes past the last slot idle along);
// the first slot's data is in a0 / b0, or already quantised in q0 / sc0 when
// `done0`; lanes k < K hold destination k in `cd`.  Every lane stores its 16
// bytes to each destination row, and the scale words go out from registers.
template <int Q>
__device__ __forceinline__ void store_token(const uint16_t *x, int t, int H, int K, uint4 a0,
                                            uint4 b0, bool done0, uint4 q0, uint32_t sc0, int cd,
                                            uint8_t *out, uint32_t *scales, int mn_stride,
                                            int mn_cap) {
    constexpr bool kFp8 = Q != EP_QUANT_NONE;
    constexpr bool kUe8m0 = Q == EP_QUANT_FP8_UE8M0 || Q == EP_QUANT_FP8_UE8M0_MN;
    const int lane = threadIdx.x & 31;
    const int G = H >> 7;
    const int row_bytes = kFp8 ? H : 2 * H;
    const int slots = kFp8 ? G * 8 : H / 8;
    const int words = kUe8m0 ? (G + 3) >> 2 : G;
    for (int j = threadIdx.x; j - lane < slots; j += blockDim.x) {
        const bool act = j < slots;
        const bool first = j == (int)threadIdx.x;
        uint4 q = q0;
        uint32_t sc = sc0;
        if (!(first && done0)) {
            uint4 a = a0, b = b0;
            if (!first) {  // passes beyond the first: loaded here
                a = b = make_uint4(0, 0, 0, 0);
                if (act) load_slot<Q>(x + (size_t)t * H, j, a, b);
            }
            q = a;
            if constexpr (kFp8) q = quant_slot<Q>(a, b, lane, sc);
        }
        for (int k = 0; k < K; ++k) {  // 16 bytes per lane to each destination
            const int d = __shfl_sync(kFullMask, cd, k);
            if (act && d >= 0) st_v4(out + (size_t)d * row_bytes + (size_t)j * 16, q);
        }
        if constexpr (kFp8)
            store_scales<Q>(scales, sc, j, lane, slots, cd, K, G, words, mn_stride, mn_cap);
    }
}

// Few tokens per SM: CTA c takes tokens c, c + gridDim.x, ...; thread i owns
// slots i, i + blockDim.x, ... (whole warps step through the passes, lanes
// past the last slot idle along) and keeps them in registers.
template <int Q>
__global__ void __launch_bounds__(512)
    direct_kernel(const uint16_t *__restrict__ x, int T, int K, int H, const int32_t *dst_row,
                  uint8_t *__restrict__ out, uint32_t *__restrict__ scales, const float *topk_w,
                  float *__restrict__ row_w, int mn_stride, int mn_cap) {
    constexpr bool kFp8 = Q != EP_QUANT_NONE;
    const int lane = threadIdx.x & 31;
    const int slots = kFp8 ? (H >> 7) * 8 : H / 8;
    const int step = gridDim.x;
    const bool weights = row_w != nullptr && threadIdx.x < K;
    const int n = cta_tokens(T, step);
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");  // see quant_kernel
    uint4 ca = make_uint4(0, 0, 0, 0), cb = ca, na = ca, nb = ca;
    const bool first_slot = (int)threadIdx.x < slots;
    if (n > 0 && first_slot) load_slot<Q>(x + (size_t)blockIdx.x * H, threadIdx.x, ca, cb);
    // x was complete before the layout started: the first token's first slot
    // is quantised while the layout may still run; dst_row is the layout's
    // output (the wait is a no-op without a programmatic edge)
    uint4 q0 = ca;
    uint32_t sc0 = 0;
    if constexpr (kFp8)
        if (n > 0) q0 = quant_slot<Q>(ca, cb, lane, sc0);
    asm volatile("griddepcontrol.wait;" ::: "memory");
    int cd = n > 0 && lane < K ? ld_dep(dst_row + (size_t)blockIdx.x * K + lane) : -1;
    float cw = n > 0 && weights ? ld_dep(topk_w + (size_t)blockIdx.x * K + lane) : 0.0f;
    // token i: the next token's slot and destinations go out first; token 0's
    // first slot was quantised before the wait (a separate copy of the step,
    // so that q0 / sc0 are dead for the others)
    auto token = [&](int i, bool first) {
        const int t = blockIdx.x + i * step;
        int nd = -1;
        float nw = 0.0f;
        if (i + 1 < n) {
            if (first_slot) load_slot<Q>(x + (size_t)(t + step) * H, threadIdx.x, na, nb);
            if (lane < K) {
                nd = ld_dep(dst_row + (size_t)(t + step) * K + lane);
                if (weights) nw = ld_dep(topk_w + (size_t)(t + step) * K + lane);
            }
        }
        if (first)
            store_token<Q>(x, t, H, K, ca, cb, true, q0, sc0, cd, out, scales, mn_stride, mn_cap);
        else
            store_token<Q>(x, t, H, K, ca, cb, false, ca, 0, cd, out, scales, mn_stride, mn_cap);
        if (weights && cd >= 0) row_w[cd] = cw;
        ca = na;
        cb = nb;
        cd = nd;
        cw = nw;
    };
    if (n > 0) token(0, true);
    for (int i = 1; i < n; ++i) token(i, false);
}

// bf16 dispatch: one warp; lane 0 drives the TMA, lanes k < K hold the
// destinations.  Token i uses stage i % stages; a stage is refilled once the
// stores of its token have read it.
__global__ void __launch_bounds__(32)
    copy_kernel(const uint16_t *__restrict__ x, int T, int K, int H, const int32_t *dst_row,
                uint8_t *__restrict__ out, const float *topk_w, float *__restrict__ row_w,
                int32_t *status, int stages, int xstage_bytes) {
    extern __shared__ __align__(128) uint8_t smem[];  // [stages] x rows
    __shared__ __align__(8) uint64_t xfull[kCopyMaxStages];
    __shared__ int s_loads[kCopyMaxStages];
    const int lane = threadIdx.x;
    const uint32_t row_bytes = 2u * (uint32_t)H;
    const int step = gridDim.x;
    const int n = cta_tokens(T, step);
    const bool weights = row_w != nullptr && lane < K;
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");  // see quant_kernel

    if (lane == 0) {
        for (int s = 0; s < stages; ++s) {
            mbar_init(&xfull[s], 1);
            s_loads[s] = s < n ? 1 : 0;
        }
        mbar_init_fence();
        for (int i = 0; i < stages && i < n; ++i)
            load_row(smem + (size_t)i * xstage_bytes, x + (size_t)(blockIdx.x + i * step) * H,
                     row_bytes, &xfull[i]);
    }
    __syncwarp();
    asm volatile("griddepcontrol.wait;" ::: "memory");  // dst_row is the layout's output
    int cd = n > 0 && lane < K ? ld_dep(dst_row + (size_t)blockIdx.x * K + lane) : -1;
    float cw = n > 0 && weights ? ld_dep(topk_w + (size_t)blockIdx.x * K + lane) : 0.0f;
    bool failed = false;
    for (int i = 0; i < n; ++i) {
        const int t = blockIdx.x + i * step;
        int nd = -1;
        float nw = 0.0f;
        if (i + 1 < n && lane < K) {
            nd = ld_dep(dst_row + (size_t)(t + step) * K + lane);
            if (weights) nw = ld_dep(topk_w + (size_t)(t + step) * K + lane);
        }
        const int s = i % stages;
        if (__any_sync(kFullMask, !mbar_wait(&xfull[s], (i / stages) & 1, nullptr))) {
            failed = true;
            break;
        }
        const uint8_t *row = smem + (size_t)s * xstage_bytes;
        for (int k = 0; k < K; ++k) {
            const int d = __shfl_sync(kFullMask, cd, k);
            if (lane == 0 && d >= 0) bulk_store(out + (size_t)d * row_bytes, row, row_bytes);
        }
        if (lane == 0) {
            bulk_commit();
            // the previous token's stage, once its stores have read it
            const int r = i - 1 + stages;
            if (i > 0 && r < n) {
                bulk_wait_read<1>();
                const int sp = (i - 1) % stages;
                load_row(smem + (size_t)sp * xstage_bytes, x + (size_t)(blockIdx.x + r * step) * H,
                         row_bytes, &xfull[sp]);
                ++s_loads[sp];
            }
        }
        if (weights && cd >= 0) row_w[cd] = cw;
        cd = nd;
        cw = nw;
    }
    if (lane == 0) {
        bulk_wait_read<0>();
        if (failed) {
            raise_status(status, EP_ERR_TIMEOUT);
            const long long t0 = clock64();
            for (int s = 0; s < stages; ++s) {
                const long long left = kWaitLimit - (clock64() - t0);
                if (s_loads[s] > 0 && (left <= 0 || !mbar_wait(&xfull[s], (s_loads[s] - 1) & 1, nullptr, left)))
                    break;
            }
        }
    }
}

// Self-test of the bounded wait: a barrier that expects 16 bytes no copy will
// ever deliver (nothing is issued, so nothing can land after the CTA exits);
// the wait must give up after `limit` SM clocks and the kernel report it.
__global__ void wait_selftest_kernel(int32_t *status, long long limit) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        mbar_init_fence();
        asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], 16;" ::"r"(smem_addr(&bar))
                     : "memory");
    }
    __syncthreads();
    const bool ok = mbar_wait(&bar, 0, nullptr, limit);
    if (__syncthreads_or(!ok) && threadIdx.x == 0) raise_status(status, EP_ERR_TIMEOUT);
}

// x stages that fit `budget` bytes beside `fixed` ones, no more than the tokens
// one CTA of two per SM would take, within [2, max_stages].
int stage_count(int T, int xstage_bytes, int fixed, int budget, int max_stages) {
    int stages = (budget - fixed) / xstage_bytes;
    const int per_cta = (T + 2 * sm_count() - 1) / (2 * sm_count());
    if (stages > per_cta) stages = per_cta;
    if (stages > max_stages) stages = max_stages;
    if (stages < 2) stages = 2;
    return stages;
}

// Persistent grid: as many CTAs as are resident at once, at most one per token.
template <typename Kern>
cudaError_t persistent_grid(Kern kern, int threads, size_t smem, int T, int &grid) {
    cudaError_t err = allow_dynamic_smem(kern, smem);
    if (err != cudaSuccess) return err;
    int per_sm = 0;
    err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, threads, smem);
    if (err != cudaSuccess) return err;
    long long g = (long long)(per_sm > 0 ? per_sm : 1) * sm_count();
    grid = (int)(g < T ? g : T);
    return cudaSuccess;
}

// MN-major scale columns: padded row space (contiguous) or padded capacity per
// expert (masked); returns the column stride, `cap` the capacity or 0.
int mn_layout(const ep_layout_t &L, int &cap) {
    const bool masked = L.kind == EP_LAYOUT_MASKED;
    const long long TK = (long long)L.num_tokens * L.num_topk;
    const long long rows_cap = masked ? (long long)L.num_experts * L.capacity
                                      : TK + (TK < L.num_experts ? TK : L.num_experts) * (L.align - 1);
    cap = masked ? L.capacity : 0;
    return masked ? (L.capacity + 3) / 4 * 4 : (int)((rows_cap + 3) / 4 * 4);
}

// Up to this many tokens per SM the direct kernel is used.
constexpr int kDirectTokensPerSm = 2;

template <int Q>
cudaError_t launch_direct(const ep_layout_t &L, const void *x, int H, void *out_rows,
                          void *out_scales, const float *topk_w, float *row_w, cudaStream_t stream) {
    const int T = L.num_tokens;
    const int slots = Q == EP_QUANT_NONE ? H / 8 : (H / 128) * 8;
    int threads = ((slots + 31) / 32) * 32;
    if (threads > 512) threads = 512;
    int grid = 0;
    cudaError_t err = persistent_grid(direct_kernel<Q>, threads, 0, T, grid);
    if (err != cudaSuccess) return err;
    int mn_cap = 0;
    const int mn_stride = mn_layout(L, mn_cap);
    return launch_kernel(direct_kernel<Q>, grid, threads, 0, stream, true,
                         static_cast<const uint16_t *>(x), T, L.num_topk, H, L.dst_row,
                         static_cast<uint8_t *>(out_rows), static_cast<uint32_t *>(out_scales),
                         topk_w, row_w, mn_stride, mn_cap);
}

template <int Q>
cudaError_t launch_quant(const ep_layout_t &L, const void *x, int H, void *out_rows,
                         void *out_scales, const float *topk_w, float *row_w, cudaStream_t stream) {
    const int T = L.num_tokens;
    const int xstage_bytes = 2 * H;  // H is a multiple of 128
    // output rows: kOutBufs, or 2 where two x stages and kOutBufs rows do not fit
    const int nob = 2 * xstage_bytes + kOutBufs * H <= kSmemMax ? kOutBufs : 2;
    const int stages = stage_count(T, xstage_bytes, nob * H, kStageBudget, kMaxStages);
    const size_t smem = (size_t)stages * xstage_bytes + (size_t)nob * H;
    int consumers = (H / 128 * 8 + 31) / 32;  // one slot of 16 elements per lane
    if (consumers > kMaxConsumerWarps) consumers = kMaxConsumerWarps;
    const int threads = 32 * (consumers + 1);
    int grid = 0;
    cudaError_t err = persistent_grid(quant_kernel<Q>, threads, smem, T, grid);
    if (err != cudaSuccess) return err;
    int mn_cap = 0;
    const int mn_stride = mn_layout(L, mn_cap);
    // programmatic dependent of the layout: the first rows load and quantise
    // while the layout kernels finish
    return launch_kernel(quant_kernel<Q>, grid, threads, smem, stream, true,
                         static_cast<const uint16_t *>(x), T, L.num_topk, H, L.dst_row,
                         static_cast<uint8_t *>(out_rows), static_cast<uint32_t *>(out_scales),
                         topk_w, row_w, L.status, mn_stride, mn_cap, stages, xstage_bytes, nob);
}

cudaError_t launch_copy(const ep_layout_t &L, const void *x, int H, void *out_rows,
                        const float *topk_w, float *row_w, cudaStream_t stream) {
    const int T = L.num_tokens;
    const int xstage_bytes = (2 * H + 127) / 128 * 128;
    const int stages = stage_count(T, xstage_bytes, 0, kCopyBudget, kCopyMaxStages);
    const size_t smem = (size_t)stages * xstage_bytes;
    int grid = 0;
    cudaError_t err = persistent_grid(copy_kernel, 32, smem, T, grid);
    if (err != cudaSuccess) return err;
    return launch_kernel(copy_kernel, grid, 32, smem, stream, true,
                         static_cast<const uint16_t *>(x), T, L.num_topk, H, L.dst_row,
                         static_cast<uint8_t *>(out_rows), topk_w, row_w, L.status, stages,
                         xstage_bytes);
}

}  // namespace

cudaError_t launch_dispatch(const ep_layout_t &L, const void *x, int H, ep_quant_t quant,
                            void *out_rows, void *out_scales, const float *topk_w,
                            float *row_w, cudaStream_t stream) {
    if (L.num_tokens == 0) return cudaSuccess;
    if (L.num_tokens <= kDirectTokensPerSm * sm_count()) {
        switch (quant) {
            case EP_QUANT_NONE:
                return launch_direct<EP_QUANT_NONE>(L, x, H, out_rows, out_scales, topk_w, row_w, stream);
            case EP_QUANT_FP8_F32:
                return launch_direct<EP_QUANT_FP8_F32>(L, x, H, out_rows, out_scales, topk_w, row_w, stream);
            case EP_QUANT_MXFP8:
                return launch_direct<EP_QUANT_MXFP8>(L, x, H, out_rows, out_scales, topk_w, row_w, stream);
            case EP_QUANT_FP8_UE8M0_MN:
                return launch_direct<EP_QUANT_FP8_UE8M0_MN>(L, x, H, out_rows, out_scales, topk_w, row_w, stream);
            default:
                return launch_direct<EP_QUANT_FP8_UE8M0>(L, x, H, out_rows, out_scales, topk_w, row_w, stream);
        }
    }
    switch (quant) {
        case EP_QUANT_NONE:
            return launch_copy(L, x, H, out_rows, topk_w, row_w, stream);
        case EP_QUANT_FP8_F32:
            return launch_quant<EP_QUANT_FP8_F32>(L, x, H, out_rows, out_scales, topk_w, row_w, stream);
        case EP_QUANT_MXFP8:
            return launch_quant<EP_QUANT_MXFP8>(L, x, H, out_rows, out_scales, topk_w, row_w, stream);
        case EP_QUANT_FP8_UE8M0_MN:
            return launch_quant<EP_QUANT_FP8_UE8M0_MN>(L, x, H, out_rows, out_scales, topk_w, row_w, stream);
        default:
            return launch_quant<EP_QUANT_FP8_UE8M0>(L, x, H, out_rows, out_scales, topk_w, row_w, stream);
    }
}

}  // namespace ep

namespace ep {

cudaError_t launch_layout_dispatch(const int32_t *topk_idx, const ep_layout_t &L,
                                   int32_t *workspace, const void *x, int H, ep_quant_t quant,
                                   void *out_rows, void *out_scales, const float *topk_w,
                                   float *row_w, cudaStream_t stream) {
    // The layout and the dispatch back to back; the dispatch is a programmatic
    // dependent of the layout, so its first rows load and quantise while the
    // layout runs.  One kernel doing both (every cluster computing the layout,
    // each CTA dispatching its slice's tokens from shared-memory destinations;
    // or every CTA recounting all entries) measured no faster at the decode
    // shapes.
    const cudaError_t err = launch_layout(topk_idx, L, workspace, stream);
    if (err != cudaSuccess) return err;
    return launch_dispatch(L, x, H, quant, out_rows, out_scales, topk_w, row_w, stream);
}

}  // namespace ep

namespace ep {

cudaError_t launch_wait_selftest(int32_t *status, long long limit_clocks, cudaStream_t stream) {
    wait_selftest_kernel<<<1, 64, 0, stream>>>(status, limit_clocks);
    return cudaGetLastError();
}

}  // namespace ep
