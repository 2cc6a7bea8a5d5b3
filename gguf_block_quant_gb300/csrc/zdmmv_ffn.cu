// zdmmv_ffn.cu -- argument checks, planning and instantiations of the
// one-launch expert FFN.
#include <cstdlib>

#include "zdmmv.h"
#include "zdmmv_ffn.cuh"

namespace zdmmv {

namespace {

template <int FGU, int LGU, int PGU, int FDN, int ST>
cudaError_t dispatch_dn_st(const FfnArgs &f, int ldn, int pdn, int smem, cudaStream_t st, bool pdl, bool query,
                           int *occ) {
#define ZDMMV_FDN(L_, P_)                                                                        \
    if (ldn == L_ && pdn == P_) {                                                                \
        if (query) {                                                                             \
            *occ = ffn_ctas_per_sm<FGU, LGU, PGU, FDN, L_, P_, ST>(smem);                        \
            return cudaSuccess;                                                                  \
        }                                                                                        \
        return launch_ffn_inst<FGU, LGU, PGU, FDN, L_, P_, ST>(f, smem, st, pdl);                \
    }
    ZDMMV_FDN(8, 1)
    ZDMMV_FDN(16, 1)
    ZDMMV_FDN(32, 1)
#undef ZDMMV_FDN
    return cudaErrorInvalidConfiguration;
}

// stages: the pipeline depth of the launch (2 or 3)
template <int FGU, int LGU, int PGU, int FDN>
cudaError_t dispatch_dn(const FfnArgs &f, int stages, int ldn, int pdn, int smem, cudaStream_t st, bool pdl,
                        bool query, int *occ) {
    if (stages == 3) return dispatch_dn_st<FGU, LGU, PGU, FDN, 3>(f, ldn, pdn, smem, st, pdl, query, occ);
    return dispatch_dn_st<FGU, LGU, PGU, FDN, 2>(f, ldn, pdn, smem, st, pdl, query, occ);
}

template <int FGU, int FDN>
cudaError_t dispatch_gu(const FfnArgs &f, int stages, int lgu, int pgu, int ldn, int pdn, int smem, cudaStream_t st,
                        bool pdl, bool query, int *occ) {
    if (lgu == 8 && pgu == 1) return dispatch_dn<FGU, 8, 1, FDN>(f, stages, ldn, pdn, smem, st, pdl, query, occ);
    if (lgu == 16 && pgu == 1) return dispatch_dn<FGU, 16, 1, FDN>(f, stages, ldn, pdn, smem, st, pdl, query, occ);
    if (lgu == 32 && pgu == 1) return dispatch_dn<FGU, 32, 1, FDN>(f, stages, ldn, pdn, smem, st, pdl, query, occ);
    if (lgu == 32 && pgu == 2) return dispatch_dn<FGU, 32, 2, FDN>(f, stages, ldn, pdn, smem, st, pdl, query, occ);
    return cudaErrorInvalidConfiguration;
}

cudaError_t dispatch(int fmt_gu, int fmt_dn, const FfnArgs &f, int stages, int lgu, int pgu, int ldn, int pdn,
                     int smem, cudaStream_t st, bool pdl, bool query, int *occ) {
    if (fmt_gu == kFmtQ4 && fmt_dn == kFmtQ8)
        return dispatch_gu<kFmtQ4, kFmtQ8>(f, stages, lgu, pgu, ldn, pdn, smem, st, pdl, query, occ);
    if (fmt_gu == kFmtQ8 && fmt_dn == kFmtQ8)
        return dispatch_gu<kFmtQ8, kFmtQ8>(f, stages, lgu, pgu, ldn, pdn, smem, st, pdl, query, occ);
    if (fmt_gu == kFmtQ4 && fmt_dn == kFmtQ4)
        return dispatch_gu<kFmtQ4, kFmtQ4>(f, stages, lgu, pgu, ldn, pdn, smem, st, pdl, query, occ);
    if (fmt_gu == kFmtQ8 && fmt_dn == kFmtQ4)
        return dispatch_gu<kFmtQ8, kFmtQ4>(f, stages, lgu, pgu, ldn, pdn, smem, st, pdl, query, occ);
    return cudaErrorInvalidConfiguration;
}

int64_t round_up_i64(int64_t v, int64_t m) { return (v + m - 1) / m * m; }

}  // namespace

size_t ffn_workspace_bytes(int n, int64_t ffn) {
    if (n <= 0 || ffn <= 0) return 0;
    const int64_t h = round_up_i64(static_cast<int64_t>(n) * ffn * 4, 256);
    return static_cast<size_t>(h + round_up_i64(8 * static_cast<int64_t>(n), 256));
}

bool ffn_shape_ok(int fmt_gu, int fmt_dn, int64_t hidden, int64_t ffn) {
    if (!tma_shape_ok(fmt_gu, hidden) || !tma_shape_ok(fmt_dn, ffn) || ffn % 128 != 0) return false;
    const TmaPlan pg = tma_plan(fmt_gu, kLayoutGguf, hidden, 2);
    const TmaPlan pd = tma_plan(fmt_dn, kLayoutGguf, ffn);
    return pg.ppl <= 2 && pd.ppl == 1;
}

namespace {
bool aligned_to(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }
}  // namespace

int ffn_entry_status(int fmt_gu, const void *w_gate, const void *w_up, int64_t gu_stride, int fmt_dn,
                     const void *w_down, int64_t dn_stride, int64_t hidden, int64_t ffn, const int32_t *idx, int n,
                     int n_experts, const void *xq, float *y, void *workspace, size_t workspace_bytes,
                     int32_t *status_dev, cudaStream_t st, bool pdl) {
    const auto bb = [](int fmt) { return fmt == kFmtQ8 ? 34 : (fmt == kFmtQ4 ? 18 : 0); };
    if (bb(fmt_gu) == 0 || bb(fmt_dn) == 0) return ZDMMV_ERR_FORMAT;
    if (hidden <= 0 || ffn <= 0 || n < 0 || n > 4096 || n_experts < 0) return ZDMMV_ERR_SHAPE;
    if (!ffn_shape_ok(fmt_gu, fmt_dn, hidden, ffn)) return ZDMMV_ERR_SHAPE;
    if (n == 0) return ZDMMV_OK;
    if (!w_gate || !w_up || !w_down || !idx || !xq || !y || !workspace) return ZDMMV_ERR_NULL;
    if (!aligned_to(w_gate, 16) || !aligned_to(w_up, 16) || !aligned_to(w_down, 16) || !aligned_to(xq, 16) ||
        !aligned_to(workspace, 256) || !aligned_to(idx, 4) || !aligned_to(y, 4) ||
        (status_dev && !aligned_to(status_dev, 4)))
        return ZDMMV_ERR_ALIGN;
    const int64_t gu_bytes = ffn * (hidden / kQK) * bb(fmt_gu);
    const int64_t dn_bytes = hidden * (ffn / kQK) * bb(fmt_dn);
    if (gu_stride < 0 || dn_stride < 0) return ZDMMV_ERR_SHAPE;
    if (n_experts > 1 && (gu_stride < gu_bytes || dn_stride < dn_bytes)) return ZDMMV_ERR_SHAPE;
    if (gu_stride % 16 || dn_stride % 16) return ZDMMV_ERR_ALIGN;
    if (workspace_bytes < ffn_workspace_bytes(n, ffn)) return ZDMMV_ERR_SIZE;
    uint32_t *fault = current_fault_word();
    if (!fault) return ZDMMV_ERR_CUDA;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return ZDMMV_ERR_CUDA;
    FfnArgs f{};
    f.w_gate = static_cast<const uint8_t *>(w_gate);
    f.w_up = static_cast<const uint8_t *>(w_up);
    f.w_down = static_cast<const uint8_t *>(w_down);
    f.gu_stride = gu_stride;
    f.dn_stride = dn_stride;
    f.idx = idx;
    f.n = n;
    f.n_experts = n_experts;
    f.status = status_dev;
    f.fault = fault;
    f.xq = static_cast<const uint8_t *>(xq);
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    const int64_t hbytes = round_up_i64(static_cast<int64_t>(n) * ffn * 4, 256);
    f.h = reinterpret_cast<float *>(ws);
    f.done = reinterpret_cast<uint32_t *>(ws + hbytes);
    f.readers = f.done + n;
    f.y = y;
    f.hidden = static_cast<int32_t>(hidden);
    f.ffn = static_cast<int32_t>(ffn);
    const cudaError_t e = launch_ffn(fmt_gu, fmt_dn, f, sms, st, pdl);
    if (e == cudaErrorNotSupported) return ZDMMV_ERR_SHAPE;  // n above what one resident grid holds
    return e == cudaSuccess ? ZDMMV_OK : ZDMMV_ERR_CUDA;
}

cudaError_t launch_ffn(int fmt_gu, int fmt_dn, FfnArgs f, int sms, cudaStream_t st, bool pdl) {
    const TmaPlan pg = tma_plan(fmt_gu, kLayoutGguf, f.hidden, 2);
    const TmaPlan pd = tma_plan(fmt_dn, kLayoutGguf, f.ffn);
    const int pitch = static_cast<int>(round_up_i64(pg.stage_bytes > pd.stage_bytes ? pg.stage_bytes : pd.stage_bytes,
                                                    256));
    const int64_t xmax = (f.hidden > f.ffn ? f.hidden : f.ffn) / kQK * 34;
    f.x_bytes_padded = static_cast<int>(round_up_i64(xmax, 128));
    f.stage_bytes = pitch;
    f.gu_tile_rows = pg.tile_rows;
    f.dn_tile_rows = pd.tile_rows;
    static const int env_stages = [] {
        const char *e = std::getenv("ZDMMV_FFN_STAGES");
        return (e && std::atoi(e) == 3) ? 3 : 2;
    }();
    static const int env_cap = [] {
        const char *e = std::getenv("ZDMMV_FFN_CTAS_PER_SM");
        const int n = e ? std::atoi(e) : 0;
        return (n >= 1 && n <= 8) ? n : 8;  // default: as many as fit (measured best)
    }();
    const int smem = kBarrierBytes + f.x_bytes_padded + env_stages * pitch;
    int occ = 0;
    cudaError_t e = dispatch(fmt_gu, fmt_dn, f, env_stages, pg.lpr, pg.ppl, pd.lpr, pd.ppl, smem, st, pdl, true,
                             &occ);
    if (e != cudaSuccess) return e;
    if (occ < 1) return cudaErrorInvalidConfiguration;
    if (occ > env_cap) occ = env_cap;
    static const int env_gu_pct = [] {
        const char *e = std::getenv("ZDMMV_FFN_GU_PERCENT");
        const int n = e ? std::atoi(e) : 0;
        return (n >= 20 && n <= 80) ? n : 60;  // measured: 50 -> 9.17, 60 -> 8.98, 67 -> 9.59 us
    }();
    // every CTA of the grid resident at once: a waiting down CTA never blocks a
    // gate/up CTA; the gate/up role takes env_gu_pct percent of the slots
    const int slots_per_expert = sms * occ / f.n;
    int gu = slots_per_expert * env_gu_pct / 100;
    int dn = slots_per_expert - gu;
    if (gu < 1 || dn < 1) return cudaErrorNotSupported;  // too many experts to be co-resident
    if (gu > f.ffn) gu = static_cast<int>(f.ffn);
    if (dn > f.hidden) dn = static_cast<int>(f.hidden);
    f.gu_per = gu;
    f.dn_per = dn;
    return dispatch(fmt_gu, fmt_dn, f, env_stages, pg.lpr, pg.ppl, pd.lpr, pd.ppl, smem, st, pdl, false, &occ);
}

}  // namespace zdmmv
