// zdmmv_ffn.cuh -- the routed experts' whole FFN in one launch: gate and up
// DMMVs with the SwiGLU epilogue, then the down DMMV of the SwiGLU output, for
// every selected expert (sm_103a).
//
// The MoE step runs the gate/up DMMV, swiglu and the down DMMV per selected
// expert ("CUDA backend for ZINC", "5. The target model & milestone ordering",
// M1) and is the largest share of the decode token (habr ZINC article,
// "Разбивка по времени"); one dispatch for all experts is the pages' remedy for
// its small per-expert matrices (habr ZINC article, "Gap analysis"; "RTX 5090:
// Batched Prefill & CUDA Graphs in ZINC", "What's next").
//
// One grid, two CTA roles:
//  * gate/up CTAs (the first n * gu_per): rows of one expert's gate and up
//    matrices, streamed pairwise into each pipeline stage as in the SwiGLU
//    epilogue of dmmv_tma_kernel; they store h = silu(gate.x) * (up.x) (fp32) to
//    the workspace and then add 1 to the expert's completion counter;
//  * down CTAs (the next n * dn_per): rows of one expert's down matrix. Their
//    producer reads the expert index and starts streaming the down weights at
//    once, overlapping the gate/up phase; the consumers wait (bounded) until the
//    expert's counter reaches gu_per, quantize h to Q8_0 blocks in shared memory
//    (the quantizer's arithmetic) and run the DMMV. The last down CTA of an
//    expert to read h resets both counters, so they are zero after every call.
// The host sizes the grid to be resident all at once (two CTAs per SM), so a
// waiting down CTA never holds the slot a gate/up CTA needs.
#pragma once

#include "zdmmv_tma.cuh"

namespace zdmmv {

struct FfnArgs {
    const uint8_t *w_gate;   // gate stack (GGUF): expert e at w_gate + e * gu_stride, ffn x hidden
    const uint8_t *w_up;     // up stack, same shape and stride
    const uint8_t *w_down;   // down stack: expert e at w_down + e * dn_stride, hidden x ffn
    int64_t gu_stride;
    int64_t dn_stride;
    const int32_t *idx;      // device int32[n]
    int32_t n;
    int32_t n_experts;
    int32_t *status;         // nullable: 1 is stored here for a bad index
    uint32_t *fault;         // device fault word
    const uint8_t *xq;       // Q8_0 blocks of the hidden activation (shared by all experts)
    float *h;                // workspace: [n][ffn] SwiGLU output
    uint32_t *done;          // workspace: [n] gate/up CTAs finished
    uint32_t *readers;       // workspace: [n] down CTAs that have read h
    float *y;                // [n][hidden] down outputs
    int32_t hidden;
    int32_t ffn;
    int32_t gu_per;          // gate/up CTAs per expert
    int32_t dn_per;          // down CTAs per expert
    int32_t gu_tile_rows;
    int32_t dn_tile_rows;
    int32_t stage_bytes;     // stage pitch (a gate/up stage holds gate then up in its halves)
    int32_t x_bytes_padded;  // shared bytes of the staged activation (the larger role's)
};

__device__ __forceinline__ uint32_t ld_acquire_gpu_u32(const uint32_t *p) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Quantize k fp32 values (k a multiple of 128) into Q8_0 blocks at xs (shared),
// with the stand-alone quantizer's arithmetic: fp32 amax, IEEE d = amax / 127 and
// 1 / d, codes round(x * id) with ties away from zero, fp16 scale (RNE). Each
// warp takes quads of blocks, 8 lanes per block, 4 values per lane.
__device__ __forceinline__ void quantize_to_smem(const float *x, int k, uint8_t *xs, int tid) {
    constexpr int kWarps = kConsumerThreads / 32;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const int sub = lane >> 3;
    const int j = lane & 7;
    const int nquads = k / 128;
    for (int qd = warp; qd < nquads; qd += kWarps) {
        const float4 v = *reinterpret_cast<const float4 *>(x + static_cast<int64_t>(4 * qd + sub) * kQK + 4 * j);
        float m = fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w)));
#pragma unroll
        for (int o = 1; o < 8; o <<= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        const float d = __fdiv_rn(m, 127.0f);
        const float id = d != 0.0f ? __frcp_rn(d) : 0.0f;
        const uint32_t c0 = static_cast<uint8_t>(static_cast<int8_t>(static_cast<int>(roundf(__fmul_rn(v.x, id)))));
        const uint32_t c1 = static_cast<uint8_t>(static_cast<int8_t>(static_cast<int>(roundf(__fmul_rn(v.y, id)))));
        const uint32_t c2 = static_cast<uint8_t>(static_cast<int8_t>(static_cast<int>(roundf(__fmul_rn(v.z, id)))));
        const uint32_t c3 = static_cast<uint8_t>(static_cast<int8_t>(static_cast<int>(roundf(__fmul_rn(v.w, id)))));
        uint8_t *blk = xs + 34 * (4 * qd + sub);
        uint16_t *dst = reinterpret_cast<uint16_t *>(blk + 2 + 4 * j);
        dst[0] = static_cast<uint16_t>(c0 | (c1 << 8));
        dst[1] = static_cast<uint16_t>(c2 | (c3 << 8));
        if (j == 0) *reinterpret_cast<unsigned short *>(blk) = __half_as_ushort(__float2half_rn(d));
    }
}

template <int FGU, int LGU, int PGU, int FDN, int LDN, int PDN, int STAGES>
__global__ void __launch_bounds__(kTmaThreads, 3) moe_ffn_kernel(const FfnArgs f) {
    extern __shared__ __align__(128) uint8_t smem[];
    uint64_t *full = reinterpret_cast<uint64_t *>(smem);
    uint64_t *empty = full + STAGES;
    uint64_t *xbar = empty + STAGES;
    uint8_t *xs = smem + kBarrierBytes;
    uint8_t *stage0 = xs + f.x_bytes_padded;

    const int tid = threadIdx.x;
    const int ngu = f.n * f.gu_per;
    const bool gu = static_cast<int>(blockIdx.x) < ngu;  // CTA-uniform role
    const int cta = gu ? static_cast<int>(blockIdx.x) : static_cast<int>(blockIdx.x) - ngu;
    const int per = gu ? f.gu_per : f.dn_per;
    const int k = cta / per;     // selected slot
    const int part = cta % per;  // this CTA's share of the expert's rows
    const int64_t rows = gu ? f.ffn : f.hidden;
    const int64_t r0 = rows * part / per;
    const int64_t r1 = rows * (part + 1) / per;  // the host keeps per <= rows: r1 > r0

    // per-role arguments of the shared tile helpers
    DmmvArgs a{};
    a.rows = rows;
    a.nb = (gu ? f.hidden : f.ffn) / kQK;
    a.tile_rows = gu ? f.gu_tile_rows : f.dn_tile_rows;
    a.stage_bytes = f.stage_bytes;
    const int T = a.tile_rows;
    const int nb = a.nb;
    const int ntiles = static_cast<int>((r1 - r0 + T - 1) / T);

    pdl_launch_dependents();
    if (tid == 0) {
#pragma unroll
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kConsumerThreads / 32);
        }
        mbar_init(xbar, 1);
        fence_barrier_init();
    }
    __syncthreads();

    if (tid >= kConsumerThreads) {
        // ------------------------------------------------------- producer
        if (tid != kConsumerThreads) return;
        pdl_wait();  // the index list and the activation may come from the preceding kernel
        const int e = f.idx[k];
        if (e < 0 || e >= f.n_experts) return;  // the consumers write NaN rows
        const uint64_t wpol = l2_evict_first_policy();
        const uint8_t *w = gu ? f.w_gate + static_cast<int64_t>(e) * f.gu_stride
                              : f.w_down + static_cast<int64_t>(e) * f.dn_stride;
        const uint8_t *w2 = gu ? f.w_up + static_cast<int64_t>(e) * f.gu_stride : nullptr;
        auto issue = [&](int t, int s) {
            if (gu)
                issue_tile<FGU, kLayoutGguf>(a, w, r0, r1, t, s, stage0, full, wpol, w2);
            else
                issue_tile<FDN, kLayoutGguf>(a, w, r0, r1, t, s, stage0, full, wpol);
        };
        // gate/up CTAs: one tile, the activation copy, then the rest of the ring
        // (this CTA's copies are served in issue order and no tile can be used
        // before the activation); down CTAs: the whole ring (their activation, h,
        // comes later from the gate/up CTAs)
        const int nring = ntiles < STAGES ? ntiles : STAGES;
        int issued = 0;
        if (gu) {
            issue(0, 0);
            issued = 1;
            const uint32_t xbytes = static_cast<uint32_t>(nb) * 34u;
            mbar_arrive_expect_tx(xbar, xbytes);
            bulk_copy_g2s(xs, f.xq, xbytes, xbar, l2_evict_last_policy());
        }
        for (; issued < nring; ++issued) issue(issued, issued);
        bool ok = true;
        for (int t = issued; t < ntiles; ++t) {
            const int s = t % STAGES;
            if (!mbar_wait(&empty[s], static_cast<uint32_t>((t / STAGES) - 1) & 1u)) {
                ok = false;
                break;
            }
            fence_proxy_async_smem();
            issue(t, s);
            issued = t + 1;
        }
        if (!ok) atomicOr(f.fault, 1u);
        for (int s = 0; s < STAGES; ++s) {
            const int t_last = (issued - 1 - s) >= 0 ? ((issued - 1 - s) / STAGES) * STAGES + s : -1;
            if (t_last >= 0) (void)mbar_wait(&full[s], static_cast<uint32_t>(t_last / STAGES) & 1u);
        }
        if (gu) (void)mbar_wait(xbar, 0);
        return;
    }

    // ---------------------------------------------------------- consumers
    const int lane = tid & 31;
    pdl_wait();
    const int e = f.idx[k];
    const bool valid = e >= 0 && e < f.n_experts;
    if (!valid && tid == 0 && f.status != nullptr) atomicExch(f.status, 1);

    if (gu) {
        constexpr int kRowsPar = kConsumerThreads / LGU;
        const int g = tid / LGU;
        const int l = tid % LGU;
        float *h = f.h + static_cast<int64_t>(k) * f.ffn;
        bool ok = true;
        if (!valid) {
            for (int64_t r = r0 + tid; r < r1; r += kConsumerThreads) h[r] = __int_as_float(0x7fc00000);
        } else {
            if (!__all_sync(0xffffffffu, mbar_wait(xbar, 0))) ok = false;
            if (ok) {
                using P = Pair<FGU, kLayoutGguf>;
                P xr[PGU];
#pragma unroll
                for (int j = 0; j < PGU; ++j) {
                    const int p = owned_pair<LGU>(l, j);
                    if (p < (nb >> 1)) {
                        uint32_t v[17];
                        load_x_pair_words_smem(smem_addr(xs), p, v);
                        xr[j].set(v);
                    }
                }
                for (int t = 0; t < ntiles && ok; ++t) {
                    const int s = t % STAGES;
                    if (!__all_sync(0xffffffffu, mbar_wait(&full[s], static_cast<uint32_t>(t / STAGES) & 1u))) {
                        ok = false;
                        break;
                    }
                    const uint32_t st = smem_addr(stage0) + static_cast<uint32_t>(s * f.stage_bytes);
                    const uint32_t st_up = st + static_cast<uint32_t>(f.stage_bytes / 2);
                    const int64_t tr0 = r0 + static_cast<int64_t>(t) * T;
                    const int nr = static_cast<int>(min(static_cast<int64_t>(T), r1 - tr0));
                    for (int base = 0; base < nr; base += kRowsPar) {
                        const int i = base + g;
                        float gv = 0.0f, uv = 0.0f;
                        if (i < nr) {
                            gv = row_partial<FGU, kLayoutGguf, LGU, PGU>(xr, st, i, T, nb, l);
                            uv = row_partial<FGU, kLayoutGguf, LGU, PGU>(xr, st_up, i, T, nb, l);
                        }
#pragma unroll
                        for (int o = LGU / 2; o > 0; o >>= 1) {
                            gv += __shfl_xor_sync(0xffffffffu, gv, o);
                            uv += __shfl_xor_sync(0xffffffffu, uv, o);
                        }
                        if (l == 0 && i < nr) h[tr0 + i] = __fmul_rn(__fdiv_rn(gv, 1.0f + expf(-gv)), uv);
                    }
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&empty[s]);
                }
            }
        }
        if (!ok && lane == 0) atomicOr(f.fault, 1u);
        // publish this CTA's rows of h (also after a fault, so no down CTA waits in vain)
        consumer_barrier();
        if (tid == 0) {
            __threadfence();
            atomicAdd(&f.done[k], 1u);
        }
        return;
    }

    // down CTA: wait until every gate/up CTA of this expert has stored its rows of h
    __shared__ int s_ready;
    if (tid == 0) {
        bool ready = ld_acquire_gpu_u32(&f.done[k]) >= static_cast<uint32_t>(f.gu_per);
        if (!ready) {
            const uint64_t t0 = global_timer_ns();
            for (uint32_t polls = 0; !ready; ++polls) {
                if (polls >= kWaitMaxPolls || global_timer_ns() - t0 > kWaitLimitNs) break;
                __nanosleep(64);
                ready = ld_acquire_gpu_u32(&f.done[k]) >= static_cast<uint32_t>(f.gu_per);
            }
        }
        s_ready = ready ? 1 : 0;
    }
    consumer_barrier();
    if (!s_ready) {
        if (tid == 0) atomicOr(f.fault, 1u);
        return;
    }
    __threadfence();  // order this thread's reads of h after the observed counter
    if (valid) quantize_to_smem(f.h + static_cast<int64_t>(k) * f.ffn, f.ffn, xs, tid);
    consumer_barrier();
    if (tid == 0) {
        // the last down CTA of this expert to read h resets the counters for the next call
        if (atomicAdd(&f.readers[k], 1u) == static_cast<uint32_t>(f.dn_per - 1)) {
            f.done[k] = 0;
            f.readers[k] = 0;
        }
    }
    float *y = f.y + static_cast<int64_t>(k) * f.hidden;
    if (!valid) {
        for (int64_t r = r0 + tid; r < r1; r += kConsumerThreads) y[r] = __int_as_float(0x7fc00000);
        return;
    }
    constexpr int kRowsPar = kConsumerThreads / LDN;
    constexpr int kRowsIlp = kTmaRowsIlp;
    const int g = tid / LDN;
    const int l = tid % LDN;
    using P = Pair<FDN, kLayoutGguf>;
    P xr[PDN];
#pragma unroll
    for (int j = 0; j < PDN; ++j) {
        const int p = owned_pair<LDN>(l, j);
        if (p < (nb >> 1)) {
            uint32_t v[17];
            load_x_pair_words_smem(smem_addr(xs), p, v);
            xr[j].set(v);
        }
    }
    for (int t = 0; t < ntiles; ++t) {
        const int s = t % STAGES;
        if (!__all_sync(0xffffffffu, mbar_wait(&full[s], static_cast<uint32_t>(t / STAGES) & 1u))) {
            if (lane == 0) atomicOr(f.fault, 1u);
            return;
        }
        const uint32_t st = smem_addr(stage0) + static_cast<uint32_t>(s * f.stage_bytes);
        const int64_t tr0 = r0 + static_cast<int64_t>(t) * T;
        const int nr = static_cast<int>(min(static_cast<int64_t>(T), r1 - tr0));
        for (int base = 0; base < nr; base += kRowsPar * kRowsIlp) {
            float acc[kRowsIlp];
#pragma unroll
            for (int r = 0; r < kRowsIlp; ++r) {
                const int i = base + r * kRowsPar + g;
                acc[r] = i < nr ? row_partial<FDN, kLayoutGguf, LDN, PDN>(xr, st, i, T, nb, l) : 0.0f;
            }
            const float part_sum = group_reduce_scatter<LDN, kRowsIlp>(acc, l);
            constexpr int kSpan = LDN / kRowsIlp;
            const int i = base + (l / kSpan) * kRowsPar + g;
            if (l % kSpan == 0 && i < nr) y[tr0 + i] = part_sum;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
    }
}

// Raise the kernel's dynamic shared-memory limit once per device.
template <int FGU, int LGU, int PGU, int FDN, int LDN, int PDN, int STAGES>
cudaError_t prepare_ffn_inst() {
    auto kern = moe_ffn_kernel<FGU, LGU, PGU, FDN, LDN, PDN, STAGES>;
    static std::atomic<bool> done[64];  // smem limit raised, per device
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!done[dev].load(std::memory_order_acquire)) {
        e = raise_dynamic_smem_limit(reinterpret_cast<const void *>(kern), dev);
        if (e != cudaSuccess) return e;
        done[dev].store(true, std::memory_order_release);
    }
    return cudaSuccess;
}

template <int FGU, int LGU, int PGU, int FDN, int LDN, int PDN, int STAGES>
cudaError_t launch_ffn_inst(const FfnArgs &f, int smem, cudaStream_t st, bool pdl) {
    auto kern = moe_ffn_kernel<FGU, LGU, PGU, FDN, LDN, PDN, STAGES>;
    cudaError_t e = prepare_ffn_inst<FGU, LGU, PGU, FDN, LDN, PDN, STAGES>();
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(f.n * (f.gu_per + f.dn_per)), 1, 1);
    cfg.blockDim = dim3(kTmaThreads, 1, 1);
    cfg.dynamicSmemBytes = static_cast<size_t>(smem);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kern, f);
}

template <int FGU, int LGU, int PGU, int FDN, int LDN, int PDN, int STAGES>
int ffn_ctas_per_sm(int smem) {
    if (prepare_ffn_inst<FGU, LGU, PGU, FDN, LDN, PDN, STAGES>() != cudaSuccess) return 0;
    int occ = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, moe_ffn_kernel<FGU, LGU, PGU, FDN, LDN, PDN, STAGES>,
                                                      kTmaThreads, static_cast<size_t>(smem)) != cudaSuccess)
        return 0;
    return occ;
}

}  // namespace zdmmv
