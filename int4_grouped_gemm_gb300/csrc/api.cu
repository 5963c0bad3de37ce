// C ABI of the int4 MoE library: argument checks, workspace layout, TMA
// descriptors and the launch sequence of each call.  See include/moe.h for
// the contract of every entry point.
#include <cudaTypedefs.h>

#include <mutex>

#include "attention.cuh"
#include "block.cuh"
#include "kernels.cuh"
#include "small_batch.cuh"


namespace moe {

static long long g_wait_limit = 4000000000LL;  // ~2 s at 2 GHz

struct DeviceInfo {
    bool ready = false;
    bool ok = false;
    int num_sms = 0;
};

static std::mutex g_mu;
static DeviceInfo g_dev[64];
static PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

static int current_device(DeviceInfo *&info) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return MOE_ERR_DEVICE;
    std::lock_guard<std::mutex> lock(g_mu);
    DeviceInfo &d = g_dev[dev];
    if (!d.ready) {
        cudaDeviceProp p{};
        if (cudaGetDeviceProperties(&p, dev) != cudaSuccess) return MOE_ERR_DEVICE;
        d.ok = (p.major == 10 && p.minor == 3);
        d.num_sms = p.multiProcessorCount;
        d.ready = true;
    }
    if (!g_encode) {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess || !fn)
            return MOE_ERR_DEVICE;
        g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
    info = &d;
    return d.ok ? MOE_OK : MOE_ERR_DEVICE;
}

static int encode_2d(CUtensorMap *map, CUtensorMapDataType type, int elem_bytes, const void *ptr, uint64_t inner,
                     uint64_t outer, uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle swz) {
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {inner * static_cast<uint64_t>(elem_bytes)};
    cuuint32_t box[2] = {box_inner, box_outer};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = g_encode(map, type, 2, const_cast<void *>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? MOE_OK : MOE_ERR_TENSOR_MAP;
}

static bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

static int check_ptr(const void *p) {
    if (!p) return MOE_ERR_NULL;
    return aligned16(p) ? MOE_OK : MOE_ERR_ALIGN;
}

static int check_shape(const moe_layer_desc *d) {
    if (!d) return MOE_ERR_NULL;
    if (d->E < 1 || d->E > 256) return MOE_ERR_SHAPE;
    if (d->k < 1 || d->k > 8 || d->k > d->E) return MOE_ERR_SHAPE;
    if (d->has_shared != 0 && d->has_shared != 1) return MOE_ERR_SHAPE;
    if (d->no_renorm != 0 && d->no_renorm != 1) return MOE_ERR_SHAPE;
    if (d->shared_gate && !d->has_shared) return MOE_ERR_SHAPE;
    if (d->group != 32 && d->group != 64) return MOE_ERR_SHAPE;
    if (d->H < 256 || d->H % 256 != 0 || d->H > 16384) return MOE_ERR_SHAPE;
    if (d->I < 128 || d->I % 128 != 0 || d->I > 4096) return MOE_ERR_SHAPE;
    return MOE_OK;
}

static int check_weights(const moe_layer_desc *d) {
    int rc;
    if ((rc = check_ptr(d->router_w))) return rc;
    if (d->router_bias && !aligned16(d->router_bias)) return MOE_ERR_ALIGN;
    if (d->shared_gate && !aligned16(d->shared_gate)) return MOE_ERR_ALIGN;
    if (d->router_split && !aligned16(d->router_split)) return MOE_ERR_ALIGN;
    const moe_qweight *ws[3] = {&d->gate, &d->up, &d->down};
    for (const moe_qweight *w : ws) {
        if ((rc = check_ptr(w->q))) return rc;
        if ((rc = check_ptr(w->scale))) return rc;
        if ((rc = check_ptr(w->bias))) return rc;
    }
    return MOE_OK;
}

static int check_tokens(const moe_layer_desc *d, int32_t T) {
    if (T < 1) return MOE_ERR_TOKENS;
    if (static_cast<int64_t>(T) * (d->k + 1) >= (int64_t(1) << 30)) return MOE_ERR_TOKENS;
    // the gate/up token copier indexes x[T][H] with 32-bit element offsets
    if (static_cast<int64_t>(T) * d->H > (int64_t(1) << 32)) return MOE_ERR_TOKENS;
    return MOE_OK;
}

static int cuda_rc(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

static cudaError_t mark(cudaEvent_t *events, int i, cudaStream_t s) {
    if (!events || !events[i]) return cudaSuccess;
    return cudaEventRecord(events[i], s);
}

// One thread waits, with the library's bounded wait, on an mbarrier that no
// thread ever arrives at; the wait must run out and record the status.
__global__ void selftest_wait_kernel(Ctrl *ctrl, long long limit) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_mbar_init();
        if (!mbar_wait(&bar, 0, limit)) record_status(&ctrl->status, MOE_ERR_TIMEOUT);
    }
}

static cudaError_t launch_selftest_wait(Ctrl *ctrl, long long limit, cudaStream_t s) {
    selftest_wait_kernel<<<1, 32, 0, s>>>(ctrl, limit);
    return cudaGetLastError();
}

}  // namespace moe

using namespace moe;

// Fixed decode scratch for moe_decode_static_scratch: one array per device,
// zero when the module loads, and from then on holding whatever the last call
// left in it.  64 KiB holds the decode scratch (control block, router sums,
// top-k, k + 1 bf16 rows of I) of E = 256, k = 8 layers up to I = 3328.
static constexpr size_t kStaticScratchBytes = 64 * 1024;
static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

static void *g_static_scratch_ptr[64];

// Look the array's device address up once per device, with that device
// current, and keep it for later calls on the same device.
static int static_scratch(char *&out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return MOE_ERR_DEVICE;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_static_scratch_ptr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess || !p) return MOE_ERR_CUDA;
        g_static_scratch_ptr[dev] = p;
    }
    out = static_cast<char *>(g_static_scratch_ptr[dev]);
    return MOE_OK;
}

// The residual stream h and the normalised layer input x of a decoder-block
// call ([T][H] bf16 each), placed after the layer's own workspace.
static size_t block_bytes(int T, int H) { return 2 * align_up(static_cast<size_t>(T) * H * 2, 256); }

static int check_block(const void *attn, const void *residual, const float *norm_w, float eps) {
    int rc;
    if ((rc = check_ptr(attn)) || (rc = check_ptr(residual)) || (rc = check_ptr(norm_w))) return rc;
    if (!(eps >= 0.0f) || !(eps < 1e30f)) return MOE_ERR_SHAPE;
    return MOE_OK;
}

extern "C" {

size_t moe_workspace_bytes(const moe_layer_desc *desc, int32_t T_max) {
    if (check_shape(desc) != MOE_OK || check_tokens(desc, T_max) != MOE_OK) return 0;
    const PrefillLayout P = prefill_layout(T_max, desc->E, desc->k, desc->H, desc->I);
    const DecodeLayout D = decode_stack_layout(desc->E, desc->k, desc->H, desc->I);
    const BatchLayout Bt = batch_layout(desc->E, desc->k, desc->H, desc->I);
    const size_t p = P.total + block_bytes(T_max, desc->H);
    const size_t b = Bt.total + block_bytes(kBatchMax, desc->H);
    size_t total = p > D.total ? p : D.total;
    return total > b ? total : b;
}

int moe_workspace_init(void *ws, size_t ws_bytes, cudaStream_t stream) {
    int rc = check_ptr(ws);
    if (rc) return rc;
    if (ws_bytes < static_cast<size_t>(kCtrlBytes)) return MOE_ERR_WORKSPACE;
    return cuda_rc(cudaMemsetAsync(ws, 0, kCtrlBytes, stream));
}

size_t moe_router_split_bytes(int32_t E, int32_t H) {
    if (E < 1 || E > 256 || H < 256 || H % 256 != 0 || H > 16384) return 0;
    return sizeof(uint16_t) * 2 * static_cast<size_t>((E + 15) / 16 * 16) * H;
}

int moe_split_router(const float *router_w, int32_t E, int32_t H, void *out, cudaStream_t stream) {
    if (!moe_router_split_bytes(E, H)) return MOE_ERR_SHAPE;
    int rc;
    if ((rc = check_ptr(router_w)) || (rc = check_ptr(out))) return rc;
    DeviceInfo *dev = nullptr;
    if ((rc = current_device(dev))) return rc;
    return cuda_rc(launch_prep(router_w, E, (E + 15) / 16 * 16, H, static_cast<__nv_bfloat16 *>(out), nullptr, 0,
                               nullptr, 0, dev->num_sms, stream));
}

int moe_routing_views_for(const moe_layer_desc *desc, int32_t T, moe_routing_views *v) {
    int rc = check_shape(desc);
    if (rc) return rc;
    if (!v) return MOE_ERR_NULL;
    if ((rc = check_tokens(desc, T))) return rc;
    const PrefillLayout L = prefill_layout(T, desc->E, desc->k, desc->H, desc->I);
    v->logits = L.logits;
    v->topk_idx = L.topk_idx;
    v->topk_w = L.topk_w;
    v->counts = L.counts;
    v->offsets = L.offsets;
    v->perm = L.perm;
    v->inv_perm = L.inv_perm;
    v->tile_group = L.tile_group;
    v->tile_row = L.tile_row;
    v->tile_rows = L.tile_rows;
    v->tile_sched = L.tile_sched;
    v->num_tiles = L.num_tiles;
    v->h = L.h;
    v->y_acc = L.y_acc;
    v->max_tiles = L.max_tiles;
    v->tile_size = kTileRows;
    return MOE_OK;
}

int moe_route_logits(const moe_layer_desc *desc, const float *logits, int32_t T, void *ws, size_t ws_bytes,
                     cudaStream_t stream) {
    int rc = check_shape(desc);
    if (rc) return rc;
    if ((rc = check_ptr(logits)) || (rc = check_ptr(ws))) return rc;
    if ((rc = check_tokens(desc, T))) return rc;
    const PrefillLayout L = prefill_layout(T, desc->E, desc->k, desc->H, desc->I);
    if (ws_bytes < L.total) return MOE_ERR_WORKSPACE;
    DeviceInfo *dev = nullptr;
    if ((rc = current_device(dev))) return rc;
    const RoutingBufs rb = routing_bufs(static_cast<char *>(ws), L);
    if (launch_zero_i32(rb.counts_blk, static_cast<int64_t>(rb.nblk) * desc->E, stream) != cudaSuccess)
        return MOE_ERR_CUDA;
    return cuda_rc(
        launch_routing_tables(nullptr, 0, logits, nullptr, T, desc->E, desc->k, desc->has_shared,
                              RouteOpts{nullptr, nullptr, desc->H, desc->no_renorm}, rb, stream));
}

static int prefill_impl(const moe_layer_desc *desc, const void *x, int32_t T, void *y, void *ws, size_t ws_bytes,
                        cudaEvent_t *events, const __nv_bfloat16 *resid, cudaStream_t stream) {
    int rc = check_shape(desc);
    if (rc) return rc;
    if ((rc = check_weights(desc))) return rc;
    if ((rc = check_ptr(x)) || (rc = check_ptr(y)) || (rc = check_ptr(ws))) return rc;
    if ((rc = check_tokens(desc, T))) return rc;
    const int E = desc->E, k = desc->k, H = desc->H, I = desc->I, G = desc->group;
    const PrefillLayout L = prefill_layout(T, E, k, H, I);
    if (ws_bytes < L.total) return MOE_ERR_WORKSPACE;
    DeviceInfo *dev = nullptr;
    if ((rc = current_device(dev))) return rc;

    char *w = static_cast<char *>(ws);
    const RoutingBufs rb = routing_bufs(w, L);
    Ctrl *ctrl = reinterpret_cast<Ctrl *>(w + L.ctrl);
    __nv_bfloat16 *h = reinterpret_cast<__nv_bfloat16 *>(w + L.h);
    float *y_acc = reinterpret_cast<float *>(w + L.y_acc);
    const int nexp = E + 1;

    __nv_bfloat16 *wr3 = reinterpret_cast<__nv_bfloat16 *>(w + L.wr3);
    float *logits_part = reinterpret_cast<float *>(w + L.logits_part);
    const int routed = T * k;
    const int ldg_h = ld_groups(H, G), ldg_i = ld_groups(I, G);
    const auto U16 = CU_TENSOR_MAP_DATA_TYPE_UINT16, U32 = CU_TENSOR_MAP_DATA_TYPE_UINT32,
               BF16 = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    const auto SW0 = CU_TENSOR_MAP_SWIZZLE_NONE, SW32 = CU_TENSOR_MAP_SWIZZLE_32B, SW64 = CU_TENSOR_MAP_SWIZZLE_64B,
               SW128 = CU_TENSOR_MAP_SWIZZLE_128B;
    const uint64_t gu_rows = static_cast<uint64_t>(nexp) * I, dn_rows = static_cast<uint64_t>(nexp) * H;

    // router: A = x tiles, B = bf16 parts of the router weights
    GemmMaps mr{}, m1{}, m2{};
    // router: the layer's split weights when the caller made them, else this
    // call's own split in the workspace
    const void *wr_src = desc->router_split ? desc->router_split : static_cast<const void *>(wr3);
    if ((rc = encode_2d(&mr.a0, BF16, 2, x, H, T, 64, 128, SW128)) ||
        (rc = encode_2d(&mr.w0, BF16, 2, wr_src, H, 2 * static_cast<uint64_t>(L.E_pad16), 64, L.E_pad16, SW128)))
        return rc;
    mr.a1 = mr.a0;
    mr.w1 = mr.s0 = mr.b0 = mr.s1 = mr.b1 = mr.w0;
    // gate/up: A = token rows gathered from x by the kernel itself (the maps
    // below are unused placeholders); B = gate rows f0..f0+127 and up rows
    // f0..f0+127 of one expert
    if ((rc = encode_2d(&m1.a0, BF16, 2, x, H, T, 64, 128, SW128)) ||
        (rc = encode_2d(&m1.a1, BF16, 2, x, H, T, 64, 128, SW128)) ||
        (rc = encode_2d(&m1.w0, U32, 4, desc->gate.q, H / 8, gu_rows, 8, 128, SW32)) ||
        (rc = encode_2d(&m1.w1, U32, 4, desc->up.q, H / 8, gu_rows, 8, 128, SW32)) ||
        (rc = encode_2d(&m1.s0, U16, 2, desc->gate.scale, ldg_h, gu_rows, 8, 128, SW0)) ||
        (rc = encode_2d(&m1.b0, U16, 2, desc->gate.bias, ldg_h, gu_rows, 8, 128, SW0)) ||
        (rc = encode_2d(&m1.s1, U16, 2, desc->up.scale, ldg_h, gu_rows, 8, 128, SW0)) ||
        (rc = encode_2d(&m1.b1, U16, 2, desc->up.bias, ldg_h, gu_rows, 8, 128, SW0)))
        return rc;
    // down: A = h rows, B = 256 down rows of one expert
    if ((rc = encode_2d(&m2.a0, BF16, 2, h, I, L.R, 64, 128, SW128)) ||
        (rc = encode_2d(&m2.w0, U32, 4, desc->down.q, I / 8, dn_rows, 16, 256, SW64)) ||
        (rc = encode_2d(&m2.s0, U16, 2, desc->down.scale, ldg_i, dn_rows, 8, 256, SW0)) ||
        (rc = encode_2d(&m2.b0, U16, 2, desc->down.bias, ldg_i, dn_rows, 8, 256, SW0)))
        return rc;
    m2.a1 = m2.a0;
    m2.w1 = m2.w0;
    m2.s1 = m2.s0;
    m2.b1 = m2.b0;

    GemmArgs ga{};
    ga.G = G;
    ga.H = H;
    ga.I = I;
    ga.T = T;
    ga.E = E;
    ga.routed_rows = routed;
    ga.E_pad16 = L.E_pad16;
    ga.rb = rb;
    ga.h = h;
    ga.x = static_cast<const __nv_bfloat16 *>(x);
    ga.y_acc = y_acc;
    ga.logits_part = logits_part;
    ga.status = &ctrl->status;
    ga.wait_limit = g_wait_limit;
    auto grid_for = [&](int units) { return dev->num_sms < units ? dev->num_sms : (units > 0 ? units : 1); };

    cudaError_t e = mark(events, 0, stream);
    if (e != cudaSuccess) return MOE_ERR_CUDA;
    // router: bf16 split of the weights unless the layer carries it, then
    // the eight partial router GEMMs on the tensor cores, whose idle warps
    // clear the expert histogram
    if (!desc->router_split &&
        launch_prep(desc->router_w, E, L.E_pad16, H, wr3, nullptr, 0, nullptr, 0, dev->num_sms, stream) != cudaSuccess)
        return MOE_ERR_CUDA;
    ga.K = H;
    ga.clear_i = rb.counts_blk;
    ga.clear_i_n = static_cast<int64_t>(rb.nblk) * E;
    if (launch_gemm(2, mr, ga, grid_for(router_units(T)), stream) != cudaSuccess) return MOE_ERR_CUDA;
    if (mark(events, 1, stream) != cudaSuccess) return MOE_ERR_CUDA;
    // routing tables
    const RouteOpts ropts{static_cast<const __nv_bfloat16 *>(x), desc->shared_gate, H, desc->no_renorm};
    if (launch_routing_tables(logits_part, L.E_pad16, nullptr, desc->router_bias, T, E, k, desc->has_shared, ropts,
                              rb, stream) != cudaSuccess)
        return MOE_ERR_CUDA;
    if (mark(events, 2, stream) != cudaSuccess) return MOE_ERR_CUDA;
    // gate/up + SwiGLU; its epilogue warps clear the fp32 combine accumulator
    // before the first unit's results arrive
    ga.K = H;
    ga.n_ntiles = I / 128;
    ga.clear_i_n = 0;
    ga.clear_f4 = reinterpret_cast<float4 *>(y_acc);
    ga.clear_f4_n = static_cast<int64_t>(T) * H / 4;
    if (launch_gemm(0, m1, ga, grid_for(L.max_tiles * ga.n_ntiles), stream) != cudaSuccess) return MOE_ERR_CUDA;
    if (mark(events, 3, stream) != cudaSuccess) return MOE_ERR_CUDA;
    // down + weighted combine
    ga.K = I;
    ga.n_ntiles = H / 256;
    ga.clear_f4_n = 0;
    if (launch_gemm(1, m2, ga, grid_for(L.max_tiles * ga.n_ntiles), stream) != cudaSuccess) return MOE_ERR_CUDA;
    if (mark(events, 4, stream) != cudaSuccess) return MOE_ERR_CUDA;
    // y = bf16 of the fp32 combine, or for a decoder block bf16(combine + h)
    const cudaError_t ce =
        resid ? launch_residual_out(y_acc, resid, static_cast<__nv_bfloat16 *>(y), static_cast<int64_t>(T) * H,
                                    dev->num_sms, stream)
              : launch_convert(y_acc, static_cast<__nv_bfloat16 *>(y), static_cast<int64_t>(T) * H, dev->num_sms,
                               stream);
    if (ce != cudaSuccess) return MOE_ERR_CUDA;
    if (mark(events, 5, stream) != cudaSuccess) return MOE_ERR_CUDA;
    return MOE_OK;
}

int moe_prefill(const moe_layer_desc *desc, const void *x, int32_t T, void *y, void *ws, size_t ws_bytes,
                cudaStream_t stream) {
    return prefill_impl(desc, x, T, y, ws, ws_bytes, nullptr, nullptr, stream);
}

int moe_prefill_profiled(const moe_layer_desc *desc, const void *x, int32_t T, void *y, void *ws, size_t ws_bytes,
                         cudaEvent_t *events, cudaStream_t stream) {
    return prefill_impl(desc, x, T, y, ws, ws_bytes, events, nullptr, stream);
}

int moe_prefill_block(const moe_layer_desc *desc, const void *attn, const void *residual, const float *norm_w,
                      float eps, int32_t T, void *out, void *ws, size_t ws_bytes, cudaStream_t stream) {
    int rc = check_shape(desc);
    if (rc) return rc;
    if ((rc = check_weights(desc))) return rc;
    if ((rc = check_block(attn, residual, norm_w, eps)) || (rc = check_ptr(out)) || (rc = check_ptr(ws))) return rc;
    if ((rc = check_tokens(desc, T))) return rc;
    const PrefillLayout L = prefill_layout(T, desc->E, desc->k, desc->H, desc->I);
    const size_t off = align_up(L.total, 256);
    if (ws_bytes < off + block_bytes(T, desc->H)) return MOE_ERR_WORKSPACE;
    DeviceInfo *dev = nullptr;
    if ((rc = current_device(dev))) return rc;
    char *w = static_cast<char *>(ws);
    __nv_bfloat16 *h = reinterpret_cast<__nv_bfloat16 *>(w + off);
    __nv_bfloat16 *x = reinterpret_cast<__nv_bfloat16 *>(w + off + block_bytes(T, desc->H) / 2);
    if (launch_residual_rmsnorm(static_cast<const __nv_bfloat16 *>(attn), static_cast<const __nv_bfloat16 *>(residual),
                                norm_w, eps, T, desc->H, h, x, stream) != cudaSuccess)
        return MOE_ERR_CUDA;
    return prefill_impl(desc, x, T, out, ws, ws_bytes, nullptr, h, stream);
}

static int decode_check(const moe_layer_desc *desc) {
    int rc = check_shape(desc);
    if (rc) return rc;
    if ((rc = check_weights(desc))) return rc;
    if (desc->H > kDecodeMaxH) return MOE_ERR_SHAPE;
    return MOE_OK;
}

static DecodeLayerPtrs decode_ptrs(const moe_layer_desc &d) {
    DecodeLayerPtrs P{};
    P.Wr = d.router_w;
    P.bias = d.router_bias;
    P.qg = d.gate.q;
    P.qu = d.up.q;
    P.qd = d.down.q;
    P.sg = d.gate.scale;
    P.bg = d.gate.bias;
    P.su = d.up.scale;
    P.bu = d.up.bias;
    P.sd = d.down.scale;
    P.bd = d.down.bias;
    P.shg = d.shared_gate;
    return P;
}

// Launches of the decode kernel for layers [0, n) of a stack whose layers
// share d0's shape; the workspace holds the layout L.  Each launch clears the
// grid-barrier counter and abort flag first.
static int decode_run(const moe_layer_desc *descs, int n, const void *x, void *y, char *w, const DecodeLayout &L,
                      int num_sms, cudaStream_t stream, float *trace = nullptr,
                      unsigned long long *tstamp = nullptr, const float *const *norm_w = nullptr, float eps = 0.f) {
    const moe_layer_desc &d0 = descs[0];
    DecodeStack a{};
    a.E = d0.E;
    a.k = d0.k;
    a.H = d0.H;
    a.I = d0.I;
    a.G = d0.group;
    a.has_shared = d0.has_shared;
    a.ldg_h = ld_groups(d0.H, d0.group);
    a.ldg_i = ld_groups(d0.I, d0.group);
    a.no_renorm = d0.no_renorm;
    a.n_total = n;
    a.x = static_cast<const __nv_bfloat16 *>(x);
    a.y = static_cast<__nv_bfloat16 *>(y);
    a.act = n > 1 ? reinterpret_cast<__nv_bfloat16 *>(w + L.act) : nullptr;
    Ctrl *ctrl = reinterpret_cast<Ctrl *>(w + L.ctrl);
    a.ctrl = ctrl;
    a.logits_part = reinterpret_cast<float *>(w + L.logits);
    a.topk_idx = reinterpret_cast<int *>(w + L.topk_idx);
    a.topk_w = reinterpret_cast<float *>(w + L.topk_w);
    a.h = reinterpret_cast<__nv_bfloat16 *>(w + L.h);
    a.racc = n > 1 ? reinterpret_cast<double *>(w + L.racc) : nullptr;  // read and written only between layers
    a.wait_limit = g_wait_limit;
    a.trace = trace;
    a.trace_ld = decode_trace_words(d0.E, d0.k);
    a.tstamp = tstamp;
    a.block_form = norm_w ? 1 : 0;
    a.eps = eps;
    for (int l0 = 0; l0 < n; l0 += kMaxStackLayers) {
        const int nl = n - l0 < kMaxStackLayers ? n - l0 : kMaxStackLayers;
        a.l0 = l0;
        a.n_layers = nl;
        for (int i = 0; i < nl; ++i) {
            a.L[i] = decode_ptrs(descs[l0 + i]);
            a.L[i].nw = norm_w ? norm_w[l0 + i] : nullptr;
        }
        a.next_Wr = l0 + nl < n ? descs[l0 + nl].router_w : nullptr;
        if (cudaMemsetAsync(&ctrl->bar, 0, 2 * sizeof(unsigned), stream) != cudaSuccess) return MOE_ERR_CUDA;
        if (launch_decode(a, num_sms, stream) != cudaSuccess) return MOE_ERR_CUDA;
    }
    return MOE_OK;
}

int moe_decode(const moe_layer_desc *desc, const void *x, void *y, void *ws, size_t ws_bytes, cudaStream_t stream) {
    int rc = decode_check(desc);
    if (rc) return rc;
    if ((rc = check_ptr(x)) || (rc = check_ptr(y)) || (rc = check_ptr(ws))) return rc;
    const DecodeLayout L = decode_layout(desc->E, desc->k, desc->I);
    if (ws_bytes < L.total) return MOE_ERR_WORKSPACE;
    DeviceInfo *dev = nullptr;
    if ((rc = current_device(dev))) return rc;
    return decode_run(desc, 1, x, y, static_cast<char *>(ws), L, dev->num_sms, stream);
}

// The small-batch layer on x (device, [B][H]); resid, if given, is added to
// the output before its rounding.  Arguments already checked.
static int batch_run(const moe_layer_desc *desc, const void *x, int32_t B, void *y, const __nv_bfloat16 *resid,
                     char *w, const BatchLayout &L, int num_sms, cudaStream_t stream) {
    BatchArgs a{};
    a.E = desc->E;
    a.k = desc->k;
    a.H = desc->H;
    a.I = desc->I;
    a.G = desc->group;
    a.B = B;
    a.has_shared = desc->has_shared;
    a.no_renorm = desc->no_renorm;
    a.ldg_h = ld_groups(desc->H, desc->group);
    a.ldg_i = ld_groups(desc->I, desc->group);
    a.S_max = L.S_max;
    a.x = static_cast<const __nv_bfloat16 *>(x);
    a.y = static_cast<__nv_bfloat16 *>(y);
    a.resid = resid;
    a.Wr = desc->router_w;
    a.bias = desc->router_bias;
    a.shg = desc->shared_gate;
    a.qg = desc->gate.q;
    a.qu = desc->up.q;
    a.qd = desc->down.q;
    a.sg = desc->gate.scale;
    a.bg = desc->gate.bias;
    a.su = desc->up.scale;
    a.bu = desc->up.bias;
    a.sd = desc->down.scale;
    a.bd = desc->down.bias;
    a.ticket = &reinterpret_cast<Ctrl *>(w + L.ctrl)->ticket;
    a.logits = reinterpret_cast<float *>(w + L.logits);
    a.slots = reinterpret_cast<int *>(w + L.slots);
    a.slot_w = reinterpret_cast<float *>(w + L.slot_w);
    a.h = reinterpret_cast<__nv_bfloat16 *>(w + L.h);
    a.o = reinterpret_cast<float *>(w + L.o);
    return cuda_rc(launch_batch(a, num_sms, stream));
}

int moe_decode_batch(const moe_layer_desc *desc, const void *x, int32_t B, void *y, void *ws, size_t ws_bytes,
                     cudaStream_t stream) {
    int rc = decode_check(desc);
    if (rc) return rc;
    if ((rc = check_ptr(x)) || (rc = check_ptr(y)) || (rc = check_ptr(ws))) return rc;
    if (B < 1 || B > kBatchMax) return MOE_ERR_TOKENS;
    const BatchLayout L = batch_layout(desc->E, desc->k, desc->H, desc->I);
    if (ws_bytes < L.total) return MOE_ERR_WORKSPACE;
    DeviceInfo *dev = nullptr;
    if ((rc = current_device(dev))) return rc;
    return batch_run(desc, x, B, y, nullptr, static_cast<char *>(ws), L, dev->num_sms, stream);
}

int moe_decode_batch_block(const moe_layer_desc *desc, const void *attn, const void *residual, const float *norm_w,
                           float eps, int32_t B, void *out, void *ws, size_t ws_bytes, cudaStream_t stream) {
    int rc = decode_check(desc);
    if (rc) return rc;
    if ((rc = check_block(attn, residual, norm_w, eps)) || (rc = check_ptr(out)) || (rc = check_ptr(ws))) return rc;
    if (B < 1 || B > kBatchMax) return MOE_ERR_TOKENS;
    const BatchLayout L = batch_layout(desc->E, desc->k, desc->H, desc->I);
    const size_t off = align_up(L.total, 256);
    if (ws_bytes < off + block_bytes(kBatchMax, desc->H)) return MOE_ERR_WORKSPACE;
    DeviceInfo *dev = nullptr;
    if ((rc = current_device(dev))) return rc;
    char *w = static_cast<char *>(ws);
    __nv_bfloat16 *h = reinterpret_cast<__nv_bfloat16 *>(w + off);
    __nv_bfloat16 *x = reinterpret_cast<__nv_bfloat16 *>(w + off + block_bytes(kBatchMax, desc->H) / 2);
    if (launch_residual_rmsnorm(static_cast<const __nv_bfloat16 *>(attn), static_cast<const __nv_bfloat16 *>(residual),
                                norm_w, eps, B, desc->H, h, x, stream) != cudaSuccess)
        return MOE_ERR_CUDA;
    return batch_run(desc, x, B, out, h, w, L, dev->num_sms, stream);
}

int moe_decode_layers(const moe_layer_desc *descs, int32_t n_layers, const void *x, void *y, void *ws,
                      size_t ws_bytes, cudaStream_t stream) {
    if (!descs) return MOE_ERR_NULL;
    if (n_layers < 1) return MOE_ERR_SHAPE;
    int rc;
    for (int l = 0; l < n_layers; ++l) {
        if ((rc = decode_check(&descs[l]))) return rc;
        const moe_layer_desc &a = descs[0], &b = descs[l];
        if (a.E != b.E || a.k != b.k || a.H != b.H || a.I != b.I || a.group != b.group ||
            a.has_shared != b.has_shared || a.no_renorm != b.no_renorm)
            return MOE_ERR_SHAPE;
    }
    if ((rc = check_ptr(x)) || (rc = check_ptr(y)) || (rc = check_ptr(ws))) return rc;
    const moe_layer_desc &d0 = descs[0];
    const DecodeLayout L = decode_stack_layout(d0.E, d0.k, d0.H, d0.I);
    if (ws_bytes < L.total) return MOE_ERR_WORKSPACE;
    DeviceInfo *dev = nullptr;
    if ((rc = current_device(dev))) return rc;
    return decode_run(descs, n_layers, x, y, static_cast<char *>(ws), L, dev->num_sms, stream);
}

int pack_int4(const float *w, int64_t rows, int32_t K, int32_t group, uint32_t *q, uint16_t *scale,
              uint16_t *bias, cudaStream_t stream) {
    int rc;
    if ((rc = check_ptr(w)) || (rc = check_ptr(q)) || (rc = check_ptr(scale)) || (rc = check_ptr(bias))) return rc;
    if (rows < 0 || K <= 0 || group <= 0 || K % 8 || group % 8 || K % group) return MOE_ERR_SHAPE;
    DeviceInfo *dev = nullptr;
    if ((rc = current_device(dev))) return rc;
    return cuda_rc(launch_pack_int4(w, rows, K, group, q, scale, bias, stream));
}

int moe_read_device_status(void *ws, cudaStream_t stream) {
    int rc = check_ptr(ws);
    if (rc) return rc;
    int status = 0;
    if (cudaMemcpyAsync(&status, ws, sizeof(int), cudaMemcpyDeviceToHost, stream) != cudaSuccess) return MOE_ERR_CUDA;
    if (cudaStreamSynchronize(stream) != cudaSuccess) return MOE_ERR_CUDA;
    if (status != 0) {
        if (cudaMemsetAsync(ws, 0, sizeof(int), stream) != cudaSuccess) return MOE_ERR_CUDA;
        if (cudaStreamSynchronize(stream) != cudaSuccess) return MOE_ERR_CUDA;
    }
    return status;
}

long long moe_set_wait_limit(long long cycles) {
    const long long prev = g_wait_limit;
    if (cycles > 0) g_wait_limit = cycles;
    return prev;
}

int moe_selftest_wait_timeout(void *ws, size_t ws_bytes, long long limit_cycles, cudaStream_t stream) {
    int rc = check_ptr(ws);
    if (rc) return rc;
    if (ws_bytes < static_cast<size_t>(kCtrlBytes)) return MOE_ERR_WORKSPACE;
    DeviceInfo *dev = nullptr;
    if ((rc = current_device(dev))) return rc;
    return cuda_rc(launch_selftest_wait(reinterpret_cast<Ctrl *>(ws), limit_cycles, stream));
}

int moe_forward_host(const moe_layer_desc *desc, const void *x_host, int32_t T, void *y_host, void *x_dev,
                     void *y_dev, void *ws, size_t ws_bytes, cudaStream_t stream) {
    int rc = check_shape(desc);
    if (rc) return rc;
    if (!x_host || !y_host) return MOE_ERR_NULL;
    if ((rc = check_tokens(desc, T))) return rc;
    const size_t bytes = static_cast<size_t>(T) * desc->H * 2;
    if (cudaMemcpyAsync(x_dev, x_host, bytes, cudaMemcpyHostToDevice, stream) != cudaSuccess) return MOE_ERR_CUDA;
    rc = T == 1 ? moe_decode(desc, x_dev, y_dev, ws, ws_bytes, stream)
                : moe_prefill(desc, x_dev, T, y_dev, ws, ws_bytes, stream);
    if (rc) return rc;
    if (cudaMemcpyAsync(y_host, y_dev, bytes, cudaMemcpyDeviceToHost, stream) != cudaSuccess) return MOE_ERR_CUDA;
    return cuda_rc(cudaStreamSynchronize(stream));
}

int moe_forward_host_stream(const moe_layer_desc *desc, const void *const *x_host, void *const *y_host, int32_t n,
                            int32_t T, void *const *x_dev, void *const *y_dev, void *ws, size_t ws_bytes,
                            cudaStream_t stream) {
    int rc = check_shape(desc);
    if (rc) return rc;
    if (n < 1) return MOE_ERR_TOKENS;
    if (!x_host || !y_host || !x_dev || !y_dev) return MOE_ERR_NULL;
    for (int i = 0; i < n; ++i)
        if (!x_host[i] || !y_host[i]) return MOE_ERR_NULL;
    for (int s = 0; s < 2; ++s)
        if ((rc = check_ptr(x_dev[s])) || (rc = check_ptr(y_dev[s]))) return rc;
    if ((rc = check_tokens(desc, T))) return rc;
    const size_t bytes = static_cast<size_t>(T) * desc->H * 2;
    cudaStream_t h2d = nullptr, d2h = nullptr;
    cudaEvent_t in_done[2] = {}, comp_done[2] = {}, out_done[2] = {};
    bool made = cudaStreamCreateWithFlags(&h2d, cudaStreamNonBlocking) == cudaSuccess &&
                cudaStreamCreateWithFlags(&d2h, cudaStreamNonBlocking) == cudaSuccess;
    for (int s = 0; s < 2 && made; ++s)
        made = cudaEventCreateWithFlags(&in_done[s], cudaEventDisableTiming) == cudaSuccess &&
               cudaEventCreateWithFlags(&comp_done[s], cudaEventDisableTiming) == cudaSuccess &&
               cudaEventCreateWithFlags(&out_done[s], cudaEventDisableTiming) == cudaSuccess;
    rc = made ? MOE_OK : MOE_ERR_CUDA;
    for (int i = 0; i < n && rc == MOE_OK; ++i) {
        const int s = i % 2;
        // x_dev[s] was last read by call i - 2's layer; y_dev[s] last copied out by its d2h
        if (i >= 2 && (cudaStreamWaitEvent(h2d, comp_done[s], 0) != cudaSuccess ||
                       cudaStreamWaitEvent(stream, out_done[s], 0) != cudaSuccess)) {
            rc = MOE_ERR_CUDA;
            break;
        }
        if (cudaMemcpyAsync(x_dev[s], x_host[i], bytes, cudaMemcpyHostToDevice, h2d) != cudaSuccess ||
            cudaEventRecord(in_done[s], h2d) != cudaSuccess || cudaStreamWaitEvent(stream, in_done[s], 0) != cudaSuccess) {
            rc = MOE_ERR_CUDA;
            break;
        }
        rc = T == 1 ? moe_decode(desc, x_dev[s], y_dev[s], ws, ws_bytes, stream)
                    : moe_prefill(desc, x_dev[s], T, y_dev[s], ws, ws_bytes, stream);
        if (rc) break;
        if (cudaEventRecord(comp_done[s], stream) != cudaSuccess || cudaStreamWaitEvent(d2h, comp_done[s], 0) != cudaSuccess ||
            cudaMemcpyAsync(y_host[i], y_dev[s], bytes, cudaMemcpyDeviceToHost, d2h) != cudaSuccess ||
            cudaEventRecord(out_done[s], d2h) != cudaSuccess)
            rc = MOE_ERR_CUDA;
    }
    // everything enqueued so far finishes before the streams and events go away
    if (h2d && cudaStreamSynchronize(h2d) != cudaSuccess) rc = rc ? rc : MOE_ERR_CUDA;
    if (cudaStreamSynchronize(stream) != cudaSuccess) rc = rc ? rc : MOE_ERR_CUDA;
    if (d2h && cudaStreamSynchronize(d2h) != cudaSuccess) rc = rc ? rc : MOE_ERR_CUDA;
    for (int s = 0; s < 2; ++s) {
        if (in_done[s]) cudaEventDestroy(in_done[s]);
        if (comp_done[s]) cudaEventDestroy(comp_done[s]);
        if (out_done[s]) cudaEventDestroy(out_done[s]);
    }
    if (h2d) cudaStreamDestroy(h2d);
    if (d2h) cudaStreamDestroy(d2h);
    return rc;
}

// ------------------------------------------------ GQA decode attention

static constexpr int kGqaMaxSms = 256;  // workspace sized for any GPU up to this many SMs

static int gqa_check(const void *q, const void *k, const void *v, int32_t Hq, int32_t Hkv, int32_t D, int32_t L,
                     int32_t L_cap, float scale, const void *out, const void *ws) {
    int rc;
    if ((rc = check_ptr(q)) || (rc = check_ptr(k)) || (rc = check_ptr(v)) || (rc = check_ptr(out)) ||
        (rc = check_ptr(ws)))
        return rc;
    if (D != 64 && D != 128) return MOE_ERR_SHAPE;
    if (Hkv < 1 || Hq < Hkv || Hq % Hkv != 0 || Hq / Hkv > 8 || Hq > 256) return MOE_ERR_SHAPE;
    if (!(scale == scale) || scale > 1e30f || scale < -1e30f) return MOE_ERR_SHAPE;
    if (L < 1 || L_cap < L || L_cap > (1 << 26)) return MOE_ERR_TOKENS;
    return MOE_OK;
}

size_t gqa_attention_workspace_bytes(int32_t Hq, int32_t Hkv, int32_t D, int32_t L) {
    if (D != 64 && D != 128) return 0;
    if (Hkv < 1 || Hq < Hkv || Hq % Hkv != 0 || Hq / Hkv > 8 || Hq > 256 || L < 1) return 0;
    const size_t packed = gqa_part_bytes(Hkv, gqa_splits(L, Hkv, kGqaMaxSms), D);
    const size_t per_head = gqa_part_bytes(Hq, gqa_splits(L, Hq, kGqaMaxSms), D);
    return packed > per_head ? packed : per_head;
}

static int gqa_run(const void *q, const void *k, const void *v, int32_t Hq, int32_t Hkv, int32_t D, int32_t L,
                   int32_t L_cap, float scale, void *out, void *ws, size_t ws_bytes, bool packed,
                   cudaStream_t stream) {
    int rc = gqa_check(q, k, v, Hq, Hkv, D, L, L_cap, scale, out, ws);
    if (rc) return rc;
    DeviceInfo *dev = nullptr;
    if ((rc = current_device(dev))) return rc;
    if (dev->num_sms > kGqaMaxSms) return MOE_ERR_DEVICE;
    GqaArgs a{};
    a.q = static_cast<const __nv_bfloat16 *>(q);
    a.k = static_cast<const __nv_bfloat16 *>(k);
    a.v = static_cast<const __nv_bfloat16 *>(v);
    a.out = static_cast<__nv_bfloat16 *>(out);
    a.Hq = Hq;
    a.Hkv = Hkv;
    a.D = D;
    a.L = L;
    a.L_cap = L_cap;
    a.group = Hq / Hkv;
    a.qpb = packed ? a.group : 1;
    a.nsplit = gqa_splits(L, Hq / a.qpb, dev->num_sms);
    a.scale = scale;
    const int blocks_y = Hq / a.qpb;
    if (ws_bytes < gqa_part_bytes(blocks_y, a.nsplit, D)) return MOE_ERR_WORKSPACE;
    a.part_o = static_cast<float *>(ws);
    a.part_ml = a.part_o + static_cast<size_t>(blocks_y) * a.nsplit * 8 * D;
    return cuda_rc(launch_gqa(a, stream));
}

int gqa_decode_attention(const void *q, const void *k_cache, const void *v_cache, int32_t Hq, int32_t Hkv, int32_t D,
                         int32_t L, int32_t L_cap, float scale, void *out, void *ws, size_t ws_bytes,
                         cudaStream_t stream) {
    return gqa_run(q, k_cache, v_cache, Hq, Hkv, D, L, L_cap, scale, out, ws, ws_bytes, true, stream);
}

int gqa_decode_attention_per_head(const void *q, const void *k_cache, const void *v_cache, int32_t Hq,
                                  int32_t Hkv, int32_t D, int32_t L, int32_t L_cap, float scale, void *out,
                                  void *ws, size_t ws_bytes, cudaStream_t stream) {
    return gqa_run(q, k_cache, v_cache, Hq, Hkv, D, L, L_cap, scale, out, ws, ws_bytes, false, stream);
}

const char *moe_status_string(int code) {
    switch (code) {
        case MOE_OK: return "ok";
        case MOE_ERR_NULL: return "a required pointer is NULL";
        case MOE_ERR_ALIGN: return "a pointer is not 16-byte aligned";
        case MOE_ERR_SHAPE: return "unsupported shape (E, k, H, I, group)";
        case MOE_ERR_TOKENS: return "token count out of range";
        case MOE_ERR_WORKSPACE: return "workspace too small";
        case MOE_ERR_CUDA: return "CUDA runtime error or failed launch";
        case MOE_ERR_TENSOR_MAP: return "TMA descriptor could not be encoded";
        case MOE_ERR_DEVICE: return "current device is not an sm_103 GPU";
        default: break;
    }
    if (code <= MOE_ERR_TIMEOUT && code > MOE_ERR_TIMEOUT - 100) return "device: a bounded wait ran out";
    return "unknown status";
}

int moe_decode_static_scratch(const moe_layer_desc *desc, const void *x, void *y, cudaStream_t stream) {
    int rc = decode_check(desc);
    if (rc) return rc;
    if ((rc = check_ptr(x)) || (rc = check_ptr(y))) return rc;
    const DecodeLayout L = decode_layout(desc->E, desc->k, desc->I);
    if (L.total > kStaticScratchBytes) return MOE_ERR_WORKSPACE;
    DeviceInfo *dev = nullptr;
    if ((rc = current_device(dev))) return rc;
    char *w = nullptr;
    if ((rc = static_scratch(w))) return rc;
    // decode_run clears the grid-barrier counter and the abort flag before
    // the launch (a call that gave up part way may have left them set); the
    // status word is left alone so that a device-side error stays readable
    // by moe_read_static_scratch_status.  Logits, top-k and h are written
    // before they are read.
    return decode_run(desc, 1, x, y, w, L, dev->num_sms, stream);
}

int moe_read_static_scratch_status(cudaStream_t stream) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return MOE_ERR_DEVICE;
    char *w = nullptr;
    {
        std::lock_guard<std::mutex> lock(g_mu);
        w = static_cast<char *>(g_static_scratch_ptr[dev]);
    }
    if (!w) return MOE_OK;  // no call on this device has used the array yet
    return moe_read_device_status(w, stream);
}

// Checks shared by the stack entry points: every layer supported by the
// decode kernel and of the first layer's shape; norm weights (if any) present
// and 16-byte aligned, eps in range.
static int stack_check(const moe_layer_desc *descs, int32_t n_layers, const float *const *norm_w, float eps) {
    if (!descs) return MOE_ERR_NULL;
    if (n_layers < 1) return MOE_ERR_SHAPE;
    int rc;
    for (int l = 0; l < n_layers; ++l) {
        if ((rc = decode_check(&descs[l]))) return rc;
        const moe_layer_desc &a = descs[0], &b = descs[l];
        if (a.E != b.E || a.k != b.k || a.H != b.H || a.I != b.I || a.group != b.group ||
            a.has_shared != b.has_shared || a.no_renorm != b.no_renorm)
            return MOE_ERR_SHAPE;
        if (norm_w && (rc = check_ptr(norm_w[l]))) return rc;
    }
    if (norm_w && (!(eps >= 0.0f) || !(eps < 1e30f))) return MOE_ERR_SHAPE;
    return MOE_OK;
}

int moe_decode_layers_traced(const moe_layer_desc *descs, const float *const *norm_w, float eps, int32_t n_layers,
                             const void *x, void *y, void *ws, size_t ws_bytes, float *routing_trace,
                             unsigned long long *time_trace, cudaStream_t stream) {
    int rc = stack_check(descs, n_layers, norm_w, eps);
    if (rc) return rc;
    if ((rc = check_ptr(x)) || (rc = check_ptr(y)) || (rc = check_ptr(ws))) return rc;
    if (routing_trace && (rc = check_ptr(routing_trace))) return rc;
    if (time_trace && (rc = check_ptr(time_trace))) return rc;
    const moe_layer_desc &d0 = descs[0];
    const DecodeLayout L = n_layers > 1 ? decode_stack_layout(d0.E, d0.k, d0.H, d0.I) : decode_layout(d0.E, d0.k, d0.I);
    if (ws_bytes < L.total) return MOE_ERR_WORKSPACE;
    DeviceInfo *dev = nullptr;
    if ((rc = current_device(dev))) return rc;
    if (dev->num_sms > kDecodeTraceMaxBlocks) return MOE_ERR_DEVICE;
    return decode_run(descs, n_layers, x, y, static_cast<char *>(ws), L, dev->num_sms, stream, routing_trace,
                      time_trace, norm_w, eps);
}

int moe_decode_layers_block(const moe_layer_desc *descs, const float *const *norm_w, float eps, int32_t n_layers,
                            const void *x, void *y, void *ws, size_t ws_bytes, cudaStream_t stream) {
    if (!norm_w) return MOE_ERR_NULL;
    int rc = stack_check(descs, n_layers, norm_w, eps);
    if (rc) return rc;
    if ((rc = check_ptr(x)) || (rc = check_ptr(y)) || (rc = check_ptr(ws))) return rc;
    const moe_layer_desc &d0 = descs[0];
    const DecodeLayout L = decode_stack_layout(d0.E, d0.k, d0.H, d0.I);
    if (ws_bytes < L.total) return MOE_ERR_WORKSPACE;
    DeviceInfo *dev = nullptr;
    if ((rc = current_device(dev))) return rc;
    return decode_run(descs, n_layers, x, y, static_cast<char *>(ws), L, dev->num_sms, stream, nullptr, nullptr,
                      norm_w, eps);
}

int moe_decode_topk_logits(const moe_layer_desc *desc, const float *logits, int32_t n, float *out,
                           cudaStream_t stream) {
    int rc = check_shape(desc);
    if (rc) return rc;
    if ((rc = check_ptr(logits)) || (rc = check_ptr(out))) return rc;
    if (n < 1) return MOE_ERR_TOKENS;
    DeviceInfo *dev = nullptr;
    if ((rc = current_device(dev))) return rc;
    DecodeStack a{};
    a.E = desc->E;
    a.k = desc->k;
    a.H = desc->H;
    a.I = desc->I;
    a.no_renorm = desc->no_renorm;
    return cuda_rc(launch_decode_topk_given(a, logits, n, out, stream));
}

int moe_batch_views_for(const moe_layer_desc *desc, moe_batch_views *v) {
    int rc = check_shape(desc);
    if (rc) return rc;
    if (!v) return MOE_ERR_NULL;
    const BatchLayout L = batch_layout(desc->E, desc->k, desc->H, desc->I);
    v->logits = L.logits;
    v->slots = L.slots;
    v->slot_w = L.slot_w;
    v->h = L.h;
    v->S_max = L.S_max;
    v->logit_ld = desc->E + 1;
    v->max_tokens = kBatchMax;
    return MOE_OK;
}

int moe_block_views_for(const moe_layer_desc *desc, int32_t T, int32_t small_batch, int64_t *h, int64_t *x) {
    int rc = check_shape(desc);
    if (rc) return rc;
    if (!h || !x) return MOE_ERR_NULL;
    size_t off, bytes;
    if (small_batch) {
        if (T < 1 || T > kBatchMax) return MOE_ERR_TOKENS;
        off = align_up(batch_layout(desc->E, desc->k, desc->H, desc->I).total, 256);
        bytes = block_bytes(kBatchMax, desc->H);
    } else {
        if ((rc = check_tokens(desc, T))) return rc;
        off = align_up(prefill_layout(T, desc->E, desc->k, desc->H, desc->I).total, 256);
        bytes = block_bytes(T, desc->H);
    }
    *h = static_cast<int64_t>(off);
    *x = static_cast<int64_t>(off + bytes / 2);
    return MOE_OK;
}

}  // extern "C"
