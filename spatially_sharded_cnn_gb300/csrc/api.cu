// api.cu -- the C ABI: argument checks, the shard plan, algorithm choice,
// workspace layout and dispatch to the kernels.  Host code only.
#include <string.h>

#include "common.cuh"

namespace hc {

std::atomic<unsigned long long> g_launches{0};

std::atomic<int> g_sm_override{0};  // hc_set_sm_count

int device_sm_count() {
    const int o = g_sm_override.load(std::memory_order_relaxed);
    if (o > 0) return o;
    static std::atomic<int> n[kMaxDevices];
    int dev = 0;
    cudaGetDevice(&dev);
    const bool cached = dev >= 0 && dev < kMaxDevices;
    int v = cached ? n[dev].load(std::memory_order_relaxed) : 0;
    if (!v) {
        if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) cudaGetLastError();
        if (v <= 0) return 1;
        if (cached) n[dev].store(v, std::memory_order_relaxed);
    }
    return v;
}

static int out_size(int in, int k, int s, int p) {
    const int span = in + 2 * p - k;
    return span < 0 ? 0 : span / s + 1;
}

static bool desc_valid(const hc_conv_desc* d) {
    if (!d) return false;
    if (d->N <= 0 || d->C_in <= 0 || d->H <= 0 || d->W <= 0 || d->C_out <= 0) return false;
    if (d->kh <= 0 || d->kw <= 0 || d->stride <= 0 || d->padding < 0 || d->groups <= 0) return false;
    if (d->num_shards <= 0 || d->num_shards_h < 0) return false;
    if (d->C_in % d->groups || d->C_out % d->groups) return false;
    if (out_size(d->H, d->kh, d->stride, d->padding) <= 0) return false;
    if (out_size(d->W, d->kw, d->stride, d->padding) <= 0) return false;
    // every tensor must stay below 2^31 elements per (n, c) plane and 2^40 overall
    const double elems = (double)d->N * d->C_in * d->H * d->W;
    return elems < 1.0e12;
}

// One dimension of the plan (Shard(3) on W, Shard(2) on H).  Block r owns
// input [r*L, (r+1)*L) and outputs [r*L/s, (r+1)*L/s) (the last block up to
// `out`); its halos are the positions outside its block that those outputs read.
static hc_status plan_1d(int in, int k, int s, int pad, int S, int out, hc_shard_extent* ext, int* widest) {
    if (S > kMaxShards) return HC_ERR_UNSUPPORTED;
    if (in % S) return HC_ERR_UNSUPPORTED;
    const int L = in / S;
    if (L % s || pad % s) return HC_ERR_UNSUPPORTED;
    *widest = 0;
    for (int r = 0; r < S; r++) {
        hc_shard_extent e;
        e.in_begin = r * L;
        e.in_end = (r + 1) * L;
        e.out_begin = r * (L / s);
        e.out_end = (r == S - 1) ? out : (r + 1) * (L / s);
        if (e.out_end > out) e.out_end = out;
        if (e.out_begin > e.out_end) e.out_begin = e.out_end;
        e.halo_left = e.halo_right = 0;
        if (e.out_end > e.out_begin) {
            const int lo = e.out_begin * s - pad;
            const int hi = (e.out_end - 1) * s - pad + k;  // one past the last position read
            if (lo < e.in_begin) e.halo_left = e.in_begin - lo;
            if (hi > e.in_end) e.halo_right = hi - e.in_end;
        }
        if (e.halo_left > L || e.halo_right > L) return HC_ERR_UNSUPPORTED;
        const int we = e.halo_left + L + e.halo_right;
        if (we > *widest) *widest = we;
        ext[r] = e;
    }
    return HC_OK;
}

hc_status make_plan(const hc_conv_desc* d, Plan* p) {
    if (!desc_valid(d)) return HC_ERR_INVALID_ARG;
    const int S = d->num_shards, s = d->stride, pad = d->padding;
    p->S = S;
    p->Wl = d->W / S;
    p->Ho = out_size(d->H, d->kh, s, pad);
    p->Wo = out_size(d->W, d->kw, s, pad);
    hc_status st = plan_1d(d->W, d->kw, s, pad, S, p->Wo, p->ext, &p->We);
    if (st) return st;
    p->Sh = d->num_shards_h > 1 ? d->num_shards_h : 1;
    if (p->Sh == 1) {  // no row neighbours: every row, no halo rows, no row crop
        p->ext_h[0] = hc_shard_extent{0, d->H, 0, 0, 0, p->Ho};
        p->Hl = d->H;
        p->Hlo = p->Ho;
        p->He = d->H;
    } else {
        if ((st = plan_1d(d->H, d->kh, s, pad, p->Sh, p->Ho, p->ext_h, &p->He))) return st;
        p->Hl = d->H / p->Sh;
        p->Hlo = p->Hl / s;
    }
    if ((long long)p->Sh * S > kMaxShards) return HC_ERR_UNSUPPORTED;
    p->Q = p->Sh * S;
    return HC_OK;
}

static bool is_s2d_conv(const hc_conv_desc* d) {
    return d->groups == 1 && d->stride >= 2 && d->kh == d->stride && d->kw == d->stride && d->padding == 0;
}

static bool aligned16(const void* q) { return ((uintptr_t)q & 15u) == 0; }

static size_t wsize(const hc_conv_desc* d) {
    return (size_t)d->C_out * (d->C_in / d->groups) * d->kh * d->kw;
}

static size_t round256(size_t b) { return (b + 255) & ~(size_t)255; }

static bool algo_supported(const hc_conv_desc* d, const Plan& p, hc_algo a) {
    switch (a) {
        case HC_ALGO_DIRECT: return true;
        case HC_ALGO_DEPTHWISE: return depthwise_supported(d, p);
        case HC_ALGO_TC_3XTF32: return tc_supported(d, p);
        case HC_ALGO_TC_BF16X6: return bf16_supported(d, p);
        default: return false;
    }
}

static hc_algo pick(const hc_conv_desc* d, const Plan& p) {
    if (depthwise_supported(d, p)) return HC_ALGO_DEPTHWISE;
    if (bf16_supported(d, p)) return HC_ALGO_TC_BF16X6;
    if (tc_supported(d, p)) return HC_ALGO_TC_3XTF32;
    return HC_ALGO_DIRECT;
}

// Workspace layout of the backward pass (bytes, each piece 256-aligned):
//   DIRECT:    [gw partials S*wsize][gb partials S*C_out]
//   DEPTHWISE: [gw partials S*C*K*K][gb partials S*C][tile partials]
//   TC_3XTF32: [gw partials][gb partials][bias scratch][NHWC hi/lo copies, weights hi/lo, split-K partials]
//   TC_BF16X6: [gw partials][gb partials][bias scratch][bf16 pieces of gy, w^T, x; split-K partials]
// reuse: the backward pass that takes x's operand copy from the forward workspace
static size_t bwd_ws_bytes(const hc_conv_desc* d, const Plan& p, hc_algo a, bool reuse = false) {
    const size_t base = round256(sizeof(float) * p.Q * wsize(d)) + round256(sizeof(float) * p.Q * d->C_out);
    size_t b = base;
    if (a == HC_ALGO_DEPTHWISE) b += round256(sizeof(float) * depthwise_bwd_ws_floats(d, p));
    if (a == HC_ALGO_TC_3XTF32) b += round256(sizeof(float) * bias_grad_ws_floats(d->C_out, p.Q)) + tc_ws_bytes(d, p, 1);
    if (a == HC_ALGO_TC_BF16X6)
        b += round256(sizeof(float) * bias_grad_ws_floats(d->C_out, p.Q)) + bf16_ws_bytes(d, p, reuse ? 2 : 1);
    // room for the patchify stem's weight-gradient slots (taken without grad_input)
    if (patchify_wgrad_supported(d, p)) {
        const size_t pw = base + round256(sizeof(float) * patchify_wgrad_ws_floats(d, p));
        if (pw > b) b = pw;
    }
    return b;
}

static size_t fwd_ws_bytes(const hc_conv_desc* d, const Plan& p, hc_algo a) {
    if (a == HC_ALGO_TC_3XTF32) return tc_ws_bytes(d, p, 0);
    if (a == HC_ALGO_TC_BF16X6) return bf16_ws_bytes(d, p, 0);
    return 0;
}

static hc_status ws_size(const hc_conv_desc* d, int pass, hc_algo a, size_t* bytes) {
    if (!bytes || pass < 0 || pass > 2) return HC_ERR_INVALID_ARG;
    Plan p;
    hc_status st = make_plan(d, &p);
    if (st) return st;
    if (a == HC_ALGO_AUTO) a = pick(d, p);
    if (!algo_supported(d, p, a)) return HC_ERR_UNSUPPORTED;
    *bytes = pass == 0 ? fwd_ws_bytes(d, p, a) : bwd_ws_bytes(d, p, a, pass == 2);
    return HC_OK;
}

// act: a GELU on the conv's input (HC_ACT_GELU_INPUT) or output
// (HC_ACT_GELU_OUTPUT), folded into the bf16-piece 1x1 convs' operand splits
static bool act_supported(const hc_conv_desc* d, hc_algo a, hc_act act) {
    if (act == HC_ACT_NONE) return true;
    return (act == HC_ACT_GELU_INPUT || act == HC_ACT_GELU_OUTPUT) && a == HC_ALGO_TC_BF16X6 && d->kh == 1 &&
           d->kw == 1 && d->stride == 1;
}

static hc_status fwd(const hc_conv_desc* d, const float* x, const float* w, const float* b, float* y, void* ws,
                     size_t ws_bytes, void* stream, hc_algo a, hc_act act = HC_ACT_NONE) {
    static thread_local Plan p;
    hc_status st = make_plan(d, &p);
    if (st) return st;
    if (!x || !w || !y || !aligned16(x) || !aligned16(w) || !aligned16(y) || (b && !aligned16(b)))
        return HC_ERR_INVALID_ARG;
    if (a == HC_ALGO_AUTO) a = pick(d, p);
    if (!algo_supported(d, p, a) || !act_supported(d, a, act)) return HC_ERR_UNSUPPORTED;
    const size_t need = fwd_ws_bytes(d, p, a);
    if (ws_bytes < need || (need && !ws) || ((uintptr_t)ws & 255)) return HC_ERR_WORKSPACE;
    cudaStream_t s = (cudaStream_t)stream;
    traced_begin(s);
    switch (a) {
        case HC_ALGO_TC_3XTF32: return launch_tc_fwd(d, p, x, w, b, y, ws, s);
        case HC_ALGO_TC_BF16X6: return launch_bf16_fwd(d, p, x, w, b, y, ws, s, act == HC_ACT_GELU_INPUT);
        case HC_ALGO_DEPTHWISE: return launch_depthwise_fwd(d, p, x, w, b, y, s);
        case HC_ALGO_DIRECT: return launch_direct_fwd(d, p, x, w, b, y, s);
        default: return HC_ERR_UNSUPPORTED;
    }
}

// fwd_ws (reuse only): the forward workspace of this desc and x, whose operand
// copy of x the backward pass reads instead of rebuilding it
static hc_status bwd(const hc_conv_desc* d, const float* x, const float* w, const float* gy, float* gx, float* gw,
                     float* gb, float* gwp_out, float* gbp_out, void* ws, size_t ws_bytes, void* stream,
                     hc_algo a, bool reuse = false, const void* fwd_ws = nullptr, size_t fwd_ws_bytes_given = 0,
                     hc_act act = HC_ACT_NONE, const float* y_pre = nullptr, const float* residual = nullptr) {
    static thread_local Plan p;
    hc_status st = make_plan(d, &p);
    if (st) return st;
    if (!x || !w || !gy || !aligned16(x) || !aligned16(w) || !aligned16(gy)) return HC_ERR_INVALID_ARG;
    for (const void* q : {(const void*)gx, (const void*)gw, (const void*)gb, (const void*)gwp_out,
                          (const void*)gbp_out})
        if (q && !aligned16(q)) return HC_ERR_INVALID_ARG;
    const bool auto_algo = a == HC_ALGO_AUTO;
    if (auto_algo) a = pick(d, p);
    if (!algo_supported(d, p, a) || !act_supported(d, a, act)) return HC_ERR_UNSUPPORTED;
    if (act == HC_ACT_GELU_OUTPUT && (!y_pre || !aligned16(y_pre))) return HC_ERR_INVALID_ARG;
    reuse = reuse && a == HC_ALGO_TC_BF16X6;  // the other families keep nothing between the passes
    if (reuse) {
        if (!fwd_ws || ((uintptr_t)fwd_ws & 255)) return HC_ERR_INVALID_ARG;
        if (fwd_ws_bytes_given < fwd_ws_bytes(d, p, a)) return HC_ERR_WORKSPACE;
    }
    const size_t need = bwd_ws_bytes(d, p, a, reuse);
    if (ws_bytes < need || (need && !ws) || ((uintptr_t)ws & 255)) return HC_ERR_WORKSPACE;
    cudaStream_t s = (cudaStream_t)stream;
    traced_begin(s);
    char* wsp = (char*)ws;
    float* gwp = (float*)wsp;
    wsp += round256(sizeof(float) * p.Q * wsize(d));
    float* gbp = (float*)wsp;
    wsp += round256(sizeof(float) * p.Q * d->C_out);
    if (gwp_out) gwp = gwp_out;
    if (gbp_out) gbp = gbp_out;
    const bool want_w = gw || gwp_out;
    const bool want_b = gb || gbp_out;
    // Weight / bias gradients alone of the patchify stem (the image needs no
    // gradient): the direct FP32 reduction reads x and grad_output once instead
    // of splitting grad_output into bf16 pieces for a 48-column GEMM.  Taken
    // when the algorithm was left to the library and the workspace holds its
    // slot table (its size follows the SM count).
    if (auto_algo && !gx && act == HC_ACT_NONE && !residual && patchify_wgrad_supported(d, p)) {
        const size_t used = (size_t)(wsp - (char*)ws);
        if (used + sizeof(float) * patchify_wgrad_ws_floats(d, p) <= ws_bytes) {
            if (!want_w && !want_b) return HC_OK;
            return launch_patchify_wgrad(d, p, x, gy, (float*)wsp, gwp, gbp, gw, gb, s);
        }
    }
    switch (a) {
        case HC_ALGO_DEPTHWISE:  // a residual gradient goes into the grad_input epilogue; the shard
                                 // partials' kernel also writes the full gradients
            st = launch_depthwise_bwd(d, p, x, w, gy, gx, (float*)wsp, gwp, gbp, want_w || want_b, s, residual, gw, gb);
            residual = nullptr;
            gw = gb = nullptr;
            break;
        case HC_ALGO_TC_3XTF32:
        case HC_ALGO_TC_BF16X6: {
            float* btmp = (float*)wsp;
            wsp += round256(sizeof(float) * bias_grad_ws_floats(d->C_out, p.Q));
            bool bias_done = false;
            // (a GELU on the output changes grad_output itself: the bias then comes from its split too)
            if (gx || want_w || (want_b && act == HC_ACT_GELU_OUTPUT)) {
                if (a == HC_ALGO_TC_BF16X6) {  // the bias partials come with grad_output's pieces
                    st = launch_bf16_bwd(d, p, x, w, gy, gx, gwp, want_w, wsp, reuse ? fwd_ws : nullptr,
                                         want_b ? gbp : nullptr, btmp, s, act == HC_ACT_GELU_INPUT,
                                         act == HC_ACT_GELU_OUTPUT ? y_pre : nullptr);
                    bias_done = true;
                } else {
                    // with the weight gradient (not space-to-depth) the bias partials come with
                    // grad_output's pieces
                    const bool fused_b = want_b && want_w && !is_s2d_conv(d);
                    st = launch_tc_bwd(d, p, x, w, gy, gx, gwp, want_w, wsp, s, fused_b ? gbp : nullptr, btmp);
                    bias_done = fused_b;
                }
                if (st) return st;
            }
            if (want_b && !bias_done)
                st = launch_bias_grad_partials(gy, gbp, d->N, d->C_out, p.Ho, p.Wo, p.S, p.Wl / d->stride, p.Sh, p.Hlo,
                                               btmp, s);
            break;
        }
        case HC_ALGO_DIRECT:  // the partials' kernel also writes the full gradients
            if (gx && (st = launch_direct_gx(d, p, w, gy, gx, s))) return st;
            if (want_w || want_b)
                st = launch_direct_partials(d, p, x, gy, want_w ? gwp : nullptr, want_b ? gbp : nullptr, s, gw, gb);
            gw = gb = nullptr;
            break;
        default: return HC_ERR_UNSUPPORTED;
    }
    if (st) return st;
    if (residual && (st = hc_add_inplace((long long)d->N * d->C_in * d->H * d->W, gx, residual, stream))) return st;
    // _Partial -> full: sum the shards' partials in shard order.
    if (gw && (st = launch_sum_rows(gwp, gw, p.Q, (long long)wsize(d), s))) return st;
    if (gb && (st = launch_sum_rows(gbp, gb, p.Q, d->C_out, s))) return st;
    return HC_OK;
}

// ---- one rank of a multi-device layout ------------------------------------
// The rank-local desc: one column block of the global desc, no shards of its
// own.  Returns HC_ERR_UNSUPPORTED unless the depthwise kernels cover it and
// its halo fits the HC_HALO_COLS margins.
static hc_status rank_local(const hc_conv_desc* d, hc_conv_desc* loc, Plan* p) {
    hc_status st = make_plan(d, p);  // validates the global split
    if (st) return st;
    if (p->Sh > 1 || d->stride != 1 || d->padding > kHaloCols) return HC_ERR_UNSUPPORTED;
    *loc = *d;
    loc->W = d->W / d->num_shards;
    loc->num_shards = 1;
    loc->num_shards_h = 1;
    if ((st = make_plan(loc, p))) return st;
    return depthwise_supported(loc, *p) ? HC_OK : HC_ERR_UNSUPPORTED;
}

static hc_status halo_layout_args(const hc_conv_desc* d, int* Wl) {
    if (!d || d->N <= 0 || d->C_in <= 0 || d->H <= 0 || d->W <= 0 || d->num_shards <= 0 || d->W % d->num_shards)
        return HC_ERR_INVALID_ARG;
    *Wl = d->W / d->num_shards;
    return *Wl % 4 ? HC_ERR_INVALID_ARG : HC_OK;
}

}  // namespace hc

using namespace hc;

extern "C" {

hc_status hc_shard_plan(const hc_conv_desc* d, hc_shard_extent* ext, int* H_out, int* W_out) {
    if (!d || !ext) return HC_ERR_INVALID_ARG;
    static thread_local Plan p;
    hc_status st = make_plan(d, &p);
    if (st) return st;
    memcpy(ext, p.ext, sizeof(hc_shard_extent) * p.S);
    if (H_out) *H_out = p.Ho;
    if (W_out) *W_out = p.Wo;
    return HC_OK;
}

hc_status hc_shard_plan_rows(const hc_conv_desc* d, hc_shard_extent* ext) {
    if (!d || !ext) return HC_ERR_INVALID_ARG;
    static thread_local Plan p;
    hc_status st = make_plan(d, &p);
    if (st) return st;
    memcpy(ext, p.ext_h, sizeof(hc_shard_extent) * p.Sh);
    return HC_OK;
}

hc_status hc_conv2d_workspace_size(const hc_conv_desc* d, int pass, size_t* bytes) {
    return ws_size(d, pass, HC_ALGO_AUTO, bytes);
}

hc_status hc_conv2d_workspace_size_algo(const hc_conv_desc* d, int pass, hc_algo algo, size_t* bytes) {
    return ws_size(d, pass, algo, bytes);
}

hc_status hc_conv2d_select(const hc_conv_desc* d, int pass, hc_algo* algo) {
    if (!algo || (pass != 0 && pass != 1)) return HC_ERR_INVALID_ARG;
    static thread_local Plan p;
    hc_status st = make_plan(d, &p);
    if (st) return st;
    *algo = pick(d, p);
    return HC_OK;
}

hc_status hc_conv2d_fwd(const hc_conv_desc* d, const float* x, const float* w, const float* bias, float* y,
                        void* ws, size_t ws_bytes, void* stream) {
    return fwd(d, x, w, bias, y, ws, ws_bytes, stream, HC_ALGO_AUTO);
}

hc_status hc_conv2d_fwd_algo(const hc_conv_desc* d, const float* x, const float* w, const float* bias, float* y,
                             void* ws, size_t ws_bytes, void* stream, hc_algo algo) {
    return fwd(d, x, w, bias, y, ws, ws_bytes, stream, algo);
}

hc_status hc_conv2d_bwd(const hc_conv_desc* d, const float* x, const float* w, const float* gy, float* gx, float* gw,
                        float* gb, float* gw_partials, float* gb_partials, void* ws, size_t ws_bytes, void* stream) {
    return bwd(d, x, w, gy, gx, gw, gb, gw_partials, gb_partials, ws, ws_bytes, stream, HC_ALGO_AUTO);
}

hc_status hc_conv2d_bwd_algo(const hc_conv_desc* d, const float* x, const float* w, const float* gy, float* gx,
                             float* gw, float* gb, float* gw_partials, float* gb_partials, void* ws, size_t ws_bytes,
                             void* stream, hc_algo algo) {
    return bwd(d, x, w, gy, gx, gw, gb, gw_partials, gb_partials, ws, ws_bytes, stream, algo);
}

hc_status hc_conv2d_bwd_reuse(const hc_conv_desc* d, const float* x, const float* w, const float* gy, float* gx,
                              float* gw, float* gb, float* gw_partials, float* gb_partials, void* ws,
                              size_t ws_bytes, const void* fwd_ws, size_t fwd_ws_bytes, void* stream, hc_algo algo) {
    return bwd(d, x, w, gy, gx, gw, gb, gw_partials, gb_partials, ws, ws_bytes, stream, algo, true, fwd_ws,
               fwd_ws_bytes);
}

hc_status hc_conv2d_bwd_residual(const hc_conv_desc* d, const float* x, const float* w, const float* gy,
                                 const float* residual, float* gx, float* gw, float* gb, float* gw_partials,
                                 float* gb_partials, void* ws, size_t ws_bytes, void* stream, hc_algo algo) {
    if (!residual || !gx || ((uintptr_t)residual & 15u) || residual == gx) return HC_ERR_INVALID_ARG;
    return bwd(d, x, w, gy, gx, gw, gb, gw_partials, gb_partials, ws, ws_bytes, stream, algo, false, nullptr, 0,
               HC_ACT_NONE, nullptr, residual);
}

hc_status hc_conv2d_fwd_act(const hc_conv_desc* d, const float* x, const float* w, const float* bias, float* y,
                            void* ws, size_t ws_bytes, void* stream, hc_algo algo, hc_act act) {
    return fwd(d, x, w, bias, y, ws, ws_bytes, stream, algo, act);
}

hc_status hc_conv2d_bwd_act(const hc_conv_desc* d, const float* x, const float* w, const float* gy, float* gx,
                            float* gw, float* gb, float* gw_partials, float* gb_partials, void* ws, size_t ws_bytes,
                            const void* fwd_ws, size_t fwd_ws_bytes, void* stream, hc_algo algo, hc_act act,
                            const float* y_pre) {
    return bwd(d, x, w, gy, gx, gw, gb, gw_partials, gb_partials, ws, ws_bytes, stream, algo, fwd_ws != nullptr,
               fwd_ws, fwd_ws_bytes, act, y_pre);
}

hc_status hc_halo_gather(const hc_conv_desc* d, const float* x, float* x_ext, void* stream) {
    static thread_local Plan p;
    hc_status st = make_plan(d, &p);
    if (st) return st;
    if (!x || !x_ext) return HC_ERR_INVALID_ARG;
    if (p.S > kMaxKernelShards || p.Sh > kMaxKernelShards) return HC_ERR_UNSUPPORTED;
    traced_begin((cudaStream_t)stream);
    return launch_halo_gather(d, p, x, x_ext, (cudaStream_t)stream);
}


hc_status hc_halo_pad(const hc_conv_desc* d, const float* x_local, float* x_pad, void* stream) {
    int Wl;
    hc_status st = halo_layout_args(d, &Wl);
    if (st) return st;
    if (!x_local || !x_pad || !aligned16(x_local) || !aligned16(x_pad)) return HC_ERR_INVALID_ARG;
    traced_begin((cudaStream_t)stream);
    return launch_halo_pad(d, Wl, x_local, x_pad, (cudaStream_t)stream);
}

hc_status hc_halo_pack(const hc_conv_desc* d, const float* x_pad, int side, float* buf, void* stream) {
    int Wl;
    hc_status st = halo_layout_args(d, &Wl);
    if (st) return st;
    if (!x_pad || !buf || (side != 0 && side != 1) || !aligned16(x_pad) || !aligned16(buf) || Wl < kHaloCols)
        return HC_ERR_INVALID_ARG;
    traced_begin((cudaStream_t)stream);
    return launch_halo_pack(d, Wl, x_pad, side, buf, (cudaStream_t)stream);
}

hc_status hc_halo_unpack(const hc_conv_desc* d, const float* buf, int side, float* x_pad, void* stream) {
    int Wl;
    hc_status st = halo_layout_args(d, &Wl);
    if (st) return st;
    if (!x_pad || (side != 0 && side != 1) || !aligned16(x_pad) || (buf && !aligned16(buf)))
        return HC_ERR_INVALID_ARG;
    traced_begin((cudaStream_t)stream);
    return launch_halo_unpack(d, Wl, buf, side, x_pad, (cudaStream_t)stream);
}

hc_status hc_conv2d_fwd_rank(const hc_conv_desc* d, const float* x_pad, const float* w, const float* bias, float* y,
                             hc_tiles tiles, void* stream) {
    static thread_local Plan p;
    hc_conv_desc loc;
    hc_status st = rank_local(d, &loc, &p);
    if (st) return st;
    if (!x_pad || !w || !y || !aligned16(x_pad) || !aligned16(w) || !aligned16(y) || (bias && !aligned16(bias)) ||
        tiles < HC_TILES_ALL || tiles > HC_TILES_EDGE)
        return HC_ERR_INVALID_ARG;
    DwLayout lay;
    lay.pitch = loc.W + 2 * kHaloCols;
    lay.xo = kHaloCols;
    lay.tiles = tiles;
    traced_begin((cudaStream_t)stream);
    return launch_depthwise_fwd(&loc, p, x_pad, w, bias, y, (cudaStream_t)stream, lay);
}

hc_status hc_conv2d_workspace_size_rank(const hc_conv_desc* d, size_t* bytes) {
    if (!bytes) return HC_ERR_INVALID_ARG;
    static thread_local Plan p;
    hc_conv_desc loc;
    hc_status st = rank_local(d, &loc, &p);
    if (st) return st;
    *bytes = sizeof(float) * depthwise_bwd_ws_floats(&loc, p);
    return HC_OK;
}

hc_status hc_conv2d_bwd_rank(const hc_conv_desc* d, const float* x_pad, const float* w, const float* gy_pad,
                             float* gx, float* gw_part, float* gb_part, void* ws, size_t ws_bytes, hc_tiles tiles,
                             void* stream) {
    static thread_local Plan p;
    hc_conv_desc loc;
    hc_status st = rank_local(d, &loc, &p);
    if (st) return st;
    if (!x_pad || !w || !gy_pad || !aligned16(x_pad) || !aligned16(w) || !aligned16(gy_pad) ||
        tiles < HC_TILES_ALL || tiles > HC_TILES_EDGE)
        return HC_ERR_INVALID_ARG;
    for (const void* q : {(const void*)gx, (const void*)gw_part, (const void*)gb_part})
        if (q && !aligned16(q)) return HC_ERR_INVALID_ARG;
    const bool want_wb = gw_part || gb_part;
    const size_t need = sizeof(float) * depthwise_bwd_ws_floats(&loc, p);
    if (want_wb && (ws_bytes < need || !ws || ((uintptr_t)ws & 15))) return HC_ERR_WORKSPACE;
    DwLayout lay;
    lay.pitch = loc.W + 2 * kHaloCols;
    lay.xo = kHaloCols;
    lay.tiles = tiles;
    lay.partials = tiles != HC_TILES_INTERIOR;
    traced_begin((cudaStream_t)stream);
    // one shard: its partials are the rank's _Partial gradients
    return launch_depthwise_bwd(&loc, p, x_pad, w, gy_pad, gx, (float*)ws, gw_part, gb_part, want_wb,
                                (cudaStream_t)stream, nullptr, nullptr, nullptr, lay);
}

hc_status hc_sum_partials(const float* parts, int count, long long n, float* out, void* stream) {
    if (!parts || !out || count <= 0 || n <= 0) return HC_ERR_INVALID_ARG;
    traced_begin((cudaStream_t)stream);
    return launch_sum_rows(parts, out, count, n, (cudaStream_t)stream);
}

hc_status hc_sync_check(void* stream) {
    if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) {
        cudaGetLastError();
        return HC_ERR_CUDA;
    }
    if (cudaGetLastError() != cudaSuccess) return HC_ERR_CUDA;
    const hc_status a = dw_take_status(), b = tc_take_status(), c = pw_take_status();
    return a ? a : b ? b : c;
}

hc_status hc_selftest_timeout(int wait_us, void* stream) {
    traced_begin((cudaStream_t)stream);
    return launch_selftest_timeout(wait_us, (cudaStream_t)stream);
}

const char* hc_status_string(hc_status s) {
    switch (s) {
        case HC_OK: return "ok";
        case HC_ERR_INVALID_ARG: return "invalid argument";
        case HC_ERR_UNSUPPORTED: return "unsupported shard plan or convolution";
        case HC_ERR_WORKSPACE: return "workspace missing or too small";
        case HC_ERR_CUDA: return "CUDA error";
        case HC_ERR_TIMEOUT: return "a kernel gave up waiting";
    }
    return "unknown status";
}

unsigned long long hc_launch_count(void) { return g_launches.load(); }

hc_status hc_set_sm_count(int sms) {
    if (sms < 0) return HC_ERR_INVALID_ARG;
    g_sm_override.store(sms, std::memory_order_relaxed);
    return HC_OK;
}

}  // extern "C"
