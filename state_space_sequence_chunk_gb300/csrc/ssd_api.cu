// ssd_api.cu -- the C ABI declared in include/ssd.h: validation, workspace
// layout and the three launches, all enqueued on the caller's stream.
#include <string.h>

#include <mutex>

#include "ssd_internal.cuh"

namespace ssd {
namespace {

constexpr size_t kAlign = 256;

size_t round_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

bool aligned16(const void* p) { return p == nullptr || ((uintptr_t)p & 15u) == 0; }

// Validate sizes; fills `p`.  Does not look at pointers.
ssd_status make_problem(const ssd_dims* d, Problem* p) {
    if (!d) return SSD_ERR_NULL;
    if (d->dtype != SSD_F32 && d->dtype != SSD_BF16) return SSD_ERR_DTYPE;
    if (d->reserved != 0) return SSD_ERR_SHAPE;
    if (d->batch < 0 || d->seqlen < 0) return SSD_ERR_SHAPE;
    if (d->nheads < 1 || d->ngroups < 1 || d->nheads % d->ngroups != 0) return SSD_ERR_SHAPE;
    if (d->chunk_size != 64 && d->chunk_size != 128 && d->chunk_size != 256) return SSD_ERR_SHAPE;
    if (d->headdim < 16 || d->headdim > 256 || d->headdim % 16 != 0) return SSD_ERR_SHAPE;
    if (d->dstate < 16 || d->dstate > 256 || d->dstate % 16 != 0) return SSD_ERR_SHAPE;
    // keep every element index and grid dimension comfortably inside int range
    if (d->batch > 65535 || d->seqlen > (1LL << 24) || d->nheads > 4096) return SSD_ERR_SHAPE;
    const int64_t tokens = d->batch * d->seqlen;
    if (tokens > 0 && tokens * d->nheads > (1LL << 31) / d->headdim) return SSD_ERR_SHAPE;
    p->b = d->batch; p->L = d->seqlen; p->H = d->nheads; p->P = d->headdim;
    p->N = d->dstate; p->G = d->ngroups; p->Q = d->chunk_size;
    p->nc = (p->L + p->Q - 1) / p->Q;
    p->Lp = p->nc * p->Q;
    p->hpg = p->H / p->G;
    p->dtype = d->dtype;
    p->esize = d->dtype == SSD_BF16 ? 2 : 4;
    if ((int64_t)p->b * p->H * p->nc * p->P * p->N > (1LL << 33)) return SSD_ERR_SHAPE;
    return SSD_OK;
}

size_t gcs_bytes(const Problem& p) { return (size_t)(p.b * p.H * p.Lp) * sizeof(float); }
size_t hid_bytes(const Problem& p) { return (size_t)(p.b * p.H * p.nc * p.P * p.N) * p.esize; }

struct Range {
    uintptr_t lo, hi;  // [lo, hi)
};
Range rng(const void* ptr, size_t bytes) {
    return Range{(uintptr_t)ptr, (uintptr_t)ptr + bytes};
}
bool overlap(Range a, Range b) {
    return a.lo != 0 && b.lo != 0 && a.hi > a.lo && b.hi > b.lo && a.lo < b.hi && b.lo < a.hi;
}

// The device must be compute capability 10.3 (the kernels are built for sm_103a).
ssd_status check_arch() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) { cudaGetLastError(); return SSD_ERR_CUDA; }
    static int cached[64];  // 0 unknown, 1 ok, 2 wrong arch
    if (dev >= 0 && dev < 64 && cached[dev] == 1) return SSD_OK;
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) {
        cudaGetLastError();
        return SSD_ERR_CUDA;
    }
    const bool ok = (major == 10 && minor == 3);
    if (dev >= 0 && dev < 64) cached[dev] = ok ? 1 : 2;
    return ok ? SSD_OK : SSD_ERR_ARCH;
}

ssd_status from_cuda(cudaError_t e) {
    if (e == cudaSuccess) return SSD_OK;
    return SSD_ERR_CUDA;
}

// One page of host memory, page-locked and mapped into every device's address
// space on first use: word `dev` is raised by a tensor-core kernel on device
// `dev` whose bounded wait gave up (report_timeout_to_host), so that the next
// call learns of it without synchronising.
constexpr int kMaxTimeoutDevices = 1024;
alignas(4096) unsigned int g_timeout_page[kMaxTimeoutDevices];
std::once_flag g_timeout_once;
unsigned int* g_timeout_dev = nullptr;   // device-usable address of g_timeout_page

unsigned int* timeout_page() {
    std::call_once(g_timeout_once, [] {
        if (cudaHostRegister(g_timeout_page, sizeof(g_timeout_page),
                             cudaHostRegisterPortable | cudaHostRegisterMapped) == cudaSuccess) {
            void* d = nullptr;
            if (cudaHostGetDevicePointer(&d, g_timeout_page, 0) == cudaSuccess)
                g_timeout_dev = static_cast<unsigned int*>(d);
        }
        cudaGetLastError();   // a failed registration only disables the early report
    });
    return g_timeout_dev;
}

// Read and clear the kernels' device error words and the host word of the
// current device; returns the error bits (~0u if they cannot be read).
unsigned int take_errors() {
    if (cudaDeviceSynchronize() != cudaSuccess) {
        cudaGetLastError();
        return ~0u;
    }
    const unsigned int a = take_fwd_pass_state_error(), b = take_compute_out_error(),
                       c = take_tf32_error();
    int dev = 0;
    if (cudaGetDevice(&dev) == cudaSuccess && dev >= 0 && dev < kMaxTimeoutDevices)
        reinterpret_cast<volatile unsigned int*>(g_timeout_page)[dev] = 0u;
    else
        cudaGetLastError();
    if (a == ~0u || b == ~0u || c == ~0u) return ~0u;
    return (a ? 1u : 0u) | (b ? 2u : 0u) | (c ? 4u : 0u);
}

// Checks made after the arguments are validated and before anything is
// enqueued: the device's compute capability, then whether a bounded wait in
// an earlier launch on this device has given up (reported once, as
// SSD_ERR_TIMEOUT; reporting it synchronises the device and clears the record).
ssd_status pre_launch() {
    const ssd_status s = check_arch();
    if (s != SSD_OK) return s;
    return timeout_pending();
}

}  // namespace

ssd_status timeout_pending() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return SSD_ERR_CUDA;
    }
    if (timeout_page() == nullptr || dev < 0 || dev >= kMaxTimeoutDevices) return SSD_OK;
    if (reinterpret_cast<volatile unsigned int*>(g_timeout_page)[dev] == 0u) return SSD_OK;
    take_errors();
    return SSD_ERR_TIMEOUT;
}

unsigned int* host_timeout_word() {
    unsigned int* page = timeout_page();
    int dev = 0;
    if (page == nullptr || cudaGetDevice(&dev) != cudaSuccess || dev < 0 ||
        dev >= kMaxTimeoutDevices) {
        cudaGetLastError();
        return nullptr;
    }
    return page + dev;
}

}  // namespace ssd

using namespace ssd;

extern "C" {

int ssd_abi_version(void) { return SSD_ABI_VERSION; }

unsigned int ssd_take_device_errors(void) { return take_errors(); }

ssd_status ssd_debug_withhold_handoffs(int on) {
    return from_cuda(set_fwd_pass_state_withhold(on ? 1u : 0u));
}

const char* ssd_status_string(ssd_status s) {
    switch (s) {
        case SSD_OK: return "ok";
        case SSD_ERR_NULL: return "a required pointer is NULL";
        case SSD_ERR_SHAPE: return "unsupported or inconsistent sizes";
        case SSD_ERR_DTYPE: return "unknown dtype code";
        case SSD_ERR_ALIGN: return "a pointer is not 16-byte aligned";
        case SSD_ERR_WORKSPACE: return "workspace smaller than ssd_fwd_workspace_bytes()";
        case SSD_ERR_ARCH: return "the current device is not compute capability 10.3 (sm_103a)";
        case SSD_ERR_CUDA: return "the CUDA runtime reported an error";
        case SSD_ERR_ALIAS: return "an output overlaps an input";
        case SSD_ERR_TIMEOUT:
            return "a bounded wait in a kernel of an earlier call gave up; that call's outputs "
                   "are undefined (nothing was enqueued by this call)";
    }
    return "unknown status";
}

ssd_status ssd_intermediate_bytes(const ssd_dims* d, size_t* gb, size_t* hb) {
    Problem p;
    ssd_status s = make_problem(d, &p);
    if (s != SSD_OK) return s;
    if (gb) *gb = gcs_bytes(p);
    if (hb) *hb = hid_bytes(p);
    return SSD_OK;
}

size_t ssd_fwd_workspace_bytes(const ssd_dims* d) {
    Problem p;
    if (make_problem(d, &p) != SSD_OK) return 0;
    if (p.b == 0 || p.L == 0) return 0;
    return 2 * round_up(gcs_bytes(p), kAlign) + round_up(hid_bytes(p), kAlign) +
           fwd_pass_state_scratch_bytes(p);
}

size_t ssd_fwd_pass_state_scratch_bytes(const ssd_dims* d) {
    Problem p;
    if (make_problem(d, &p) != SSD_OK) return 0;
    return fwd_pass_state_scratch_bytes(p);
}

ssd_status ssd_chunk_cumsum(const ssd_dims* d, const float* dt, const float* A, float* Gcs,
                            float* dtT, void* stream) {
    Problem p;
    ssd_status s = make_problem(d, &p);
    if (s != SSD_OK) return s;
    if (p.b == 0 || p.L == 0) return SSD_OK;
    if (!dt || !A || !Gcs || !dtT) return SSD_ERR_NULL;
    if (!aligned16(dt) || !aligned16(A) || !aligned16(Gcs) || !aligned16(dtT)) return SSD_ERR_ALIGN;
    const size_t gb = gcs_bytes(p);
    const Range in[] = {rng(dt, (size_t)(p.b * p.L * p.H) * 4), rng(A, (size_t)p.H * 4)};
    for (const Range& r : in)
        if (overlap(r, rng(Gcs, gb)) || overlap(r, rng(dtT, gb))) return SSD_ERR_ALIAS;
    if (overlap(rng(Gcs, gb), rng(dtT, gb))) return SSD_ERR_ALIAS;
    if ((s = pre_launch()) != SSD_OK) return s;
    return from_cuda(launch_chunk_cumsum(p, dt, A, Gcs, dtT, nullptr, 0, (cudaStream_t)stream));
}

ssd_status ssd_fwd_pass_state(const ssd_dims* d, const void* x, const void* B, const float* Gcs,
                              const float* dtT, const float* init_state, void* hiddens,
                              float* final_state, void* scratch, size_t scratch_bytes,
                              void* stream) {
    Problem p;
    ssd_status s = make_problem(d, &p);
    if (s != SSD_OK) return s;
    const size_t sbytes = (size_t)(p.b * p.H * p.P * p.N) * 4;
    if (p.b == 0) return SSD_OK;
    if (p.L == 0) {
        if (!final_state) return SSD_OK;
        if (!aligned16(final_state) || !aligned16(init_state)) return SSD_ERR_ALIGN;
        if ((s = pre_launch()) != SSD_OK) return s;
        cudaError_t e = init_state
            ? (init_state == final_state ? cudaSuccess
                                         : cudaMemcpyAsync(final_state, init_state, sbytes,
                                                           cudaMemcpyDeviceToDevice,
                                                           (cudaStream_t)stream))
            : cudaMemsetAsync(final_state, 0, sbytes, (cudaStream_t)stream);
        return from_cuda(e);
    }
    if (!x || !B || !Gcs || !dtT || !hiddens) return SSD_ERR_NULL;
    const size_t need = fwd_pass_state_scratch_bytes(p);
    if (need > 0 && !scratch) return SSD_ERR_NULL;
    if (scratch_bytes < need) return SSD_ERR_WORKSPACE;
    if (!aligned16(x) || !aligned16(B) || !aligned16(Gcs) || !aligned16(dtT) ||
        !aligned16(init_state) || !aligned16(hiddens) || !aligned16(final_state) ||
        !aligned16(scratch))
        return SSD_ERR_ALIGN;
    const size_t es = (size_t)p.esize, gb = gcs_bytes(p);
    const Range in[] = {rng(x, (size_t)(p.b * p.L * p.H * p.P) * es),
                        rng(B, (size_t)(p.b * p.L * p.G * p.N) * es), rng(Gcs, gb), rng(dtT, gb),
                        rng(init_state, sbytes)};
    const Range hid = rng(hiddens, hid_bytes(p)), fin = rng(final_state, sbytes);
    for (int i = 0; i < 5; ++i) {
        if (overlap(in[i], hid)) return SSD_ERR_ALIAS;
        if (i < 4 && overlap(in[i], fin)) return SSD_ERR_ALIAS;
    }
    if (init_state && final_state && init_state != final_state && overlap(in[4], fin))
        return SSD_ERR_ALIAS;
    if (overlap(hid, fin)) return SSD_ERR_ALIAS;
    const Range scr = rng(need > 0 ? scratch : nullptr, need);
    for (const Range& r : in)
        if (overlap(r, scr)) return SSD_ERR_ALIAS;
    if (overlap(scr, hid) || overlap(scr, fin)) return SSD_ERR_ALIAS;
    if ((s = pre_launch()) != SSD_OK) return s;
    return from_cuda(launch_fwd_pass_state(p, x, B, Gcs, dtT, init_state, hiddens, final_state,
                                           scratch, false, (cudaStream_t)stream));
}

ssd_status ssd_compute_out(const ssd_dims* d, const void* x, const void* B, const void* C,
                           const float* Gcs, const float* dtT, const void* hiddens, const float* D,
                           void* y, void* stream) {
    Problem p;
    ssd_status s = make_problem(d, &p);
    if (s != SSD_OK) return s;
    if (p.b == 0 || p.L == 0) return SSD_OK;
    if (!x || !B || !C || !Gcs || !dtT || !hiddens || !y) return SSD_ERR_NULL;
    if (!aligned16(x) || !aligned16(B) || !aligned16(C) || !aligned16(Gcs) || !aligned16(dtT) ||
        !aligned16(hiddens) || !aligned16(D) || !aligned16(y))
        return SSD_ERR_ALIGN;
    const size_t es = (size_t)p.esize, gb = gcs_bytes(p);
    const size_t xb = (size_t)(p.b * p.L * p.H * p.P) * es;
    const size_t bcb = (size_t)(p.b * p.L * p.G * p.N) * es;
    const Range in[] = {rng(x, xb), rng(B, bcb), rng(C, bcb), rng(Gcs, gb), rng(dtT, gb),
                        rng(hiddens, hid_bytes(p)), rng(D, (size_t)p.H * 4)};
    for (const Range& r : in)
        if (overlap(r, rng(y, xb))) return SSD_ERR_ALIAS;
    if ((s = pre_launch()) != SSD_OK) return s;
    return from_cuda(launch_compute_out(p, x, B, C, Gcs, dtT, hiddens, D, y, (cudaStream_t)stream));
}

ssd_status ssd_causal_conv1d(const ssd_conv_dims* d, const void* x, const float* weight,
                             const float* bias, void* out, void* stream) {
    if (!d) return SSD_ERR_NULL;
    if (d->dtype != SSD_F32 && d->dtype != SSD_BF16) return SSD_ERR_DTYPE;
    if (d->reserved != 0 || d->batch < 0 || d->batch > 65535 || d->dim < 1 || d->dim > 65535 ||
        d->seqlen < 0 || d->seqlen > (1LL << 30) || d->width < 1 || d->width > 8)
        return SSD_ERR_SHAPE;
    if (d->batch * d->dim > (1LL << 31) / (d->seqlen > 0 ? d->seqlen : 1)) return SSD_ERR_SHAPE;
    ConvProblem p;
    p.b = d->batch; p.dim = d->dim; p.L = d->seqlen; p.W = d->width;
    p.dtype = d->dtype;
    p.esize = d->dtype == SSD_BF16 ? 2 : 4;
    if (p.b == 0 || p.L == 0) return SSD_OK;
    if (!x || !weight || !out) return SSD_ERR_NULL;
    if (!aligned16(x) || !aligned16(weight) || !aligned16(bias) || !aligned16(out))
        return SSD_ERR_ALIGN;
    const size_t xb = (size_t)(p.b * p.dim * p.L) * p.esize;
    const Range orr = rng(out, xb);
    if (overlap(orr, rng(x, xb)) || overlap(orr, rng(weight, (size_t)(p.dim * p.W) * 4)) ||
        overlap(orr, rng(bias, (size_t)p.dim * 4)))
        return SSD_ERR_ALIAS;
    ssd_status s = pre_launch();
    if (s != SSD_OK) return s;
    return from_cuda(launch_causal_conv1d(p, x, weight, bias, out, (cudaStream_t)stream));
}

static ssd_status make_gdn(const ssd_gdn_dims* d, GdnProblem* p) {
    if (!d) return SSD_ERR_NULL;
    if (d->dtype != SSD_F32) return SSD_ERR_DTYPE;
    if (d->reserved != 0 || d->batch < 0 || d->seqlen < 0 || d->nheads < 1 || d->kdim < 4 ||
        d->kdim > 128 || d->kdim % 4 != 0 || d->vdim < 1 || d->vdim > 128 ||
        (d->chunk != 16 && d->chunk != 32 && d->chunk != 64))
        return SSD_ERR_SHAPE;
    p->B = d->batch; p->T = d->seqlen; p->H = d->nheads; p->K = d->kdim; p->V = d->vdim;
    p->C = d->chunk;
    p->NT = (p->T + p->C - 1) / p->C;
    if (p->NT > 65535 || p->B * p->H > (1LL << 30) || p->B * p->T * p->H * 128 > (1LL << 40))
        return SSD_ERR_SHAPE;
    return SSD_OK;
}

ssd_status ssd_gdn_chunk_fwd_h(const ssd_gdn_dims* d, const float* k, const float* w,
                               const float* u, const float* g, const float* h0, float* h,
                               float* v_new, float* final_state, void* stream) {
    GdnProblem p;
    ssd_status s = make_gdn(d, &p);
    if (s != SSD_OK) return s;
    if (p.B == 0) return SSD_OK;
    // with no tokens the inputs are not read: only the state passes through
    if (p.T > 0 && (!k || !w || !u || !g || !h || !v_new)) return SSD_ERR_NULL;
    if (!aligned16(k) || !aligned16(w) || !aligned16(u) || !aligned16(g) || !aligned16(h0) ||
        !aligned16(h) || !aligned16(v_new) || !aligned16(final_state))
        return SSD_ERR_ALIGN;
    const size_t kb = (size_t)(p.B * p.T * p.H * p.K) * 4, vb = (size_t)(p.B * p.T * p.H * p.V) * 4;
    const size_t sb = (size_t)(p.B * p.H * p.K * p.V) * 4;
    const Range in[] = {rng(k, kb), rng(w, kb), rng(u, vb), rng(g, (size_t)(p.B * p.T * p.H) * 4),
                        rng(h0, sb)};
    const Range out[] = {rng(h, sb * (size_t)p.NT), rng(v_new, vb), rng(final_state, sb)};
    for (const Range& o : out) {
        for (const Range& r : in)
            if (overlap(o, r)) return SSD_ERR_ALIAS;
    }
    if (overlap(out[0], out[1]) || overlap(out[0], out[2]) || overlap(out[1], out[2]))
        return SSD_ERR_ALIAS;
    if ((s = pre_launch()) != SSD_OK) return s;
    return from_cuda(launch_gdn_fwd_h(p, k, w, u, g, h0, h, v_new, final_state,
                                      (cudaStream_t)stream));
}

ssd_status ssd_gdn_chunk_fwd_o(const ssd_gdn_dims* d, const float* q, const float* k,
                               const float* v_new, const float* h, const float* g, float* o,
                               void* stream) {
    GdnProblem p;
    ssd_status s = make_gdn(d, &p);
    if (s != SSD_OK) return s;
    if (p.B == 0 || p.T == 0) return SSD_OK;
    if (!q || !k || !v_new || !h || !g || !o) return SSD_ERR_NULL;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v_new) || !aligned16(h) || !aligned16(g) ||
        !aligned16(o))
        return SSD_ERR_ALIGN;
    const size_t kb = (size_t)(p.B * p.T * p.H * p.K) * 4, vb = (size_t)(p.B * p.T * p.H * p.V) * 4;
    const size_t hb = (size_t)(p.B * p.H * p.NT * p.K * p.V) * 4;
    const Range in[] = {rng(q, kb), rng(k, kb), rng(v_new, vb), rng(h, hb),
                        rng(g, (size_t)(p.B * p.T * p.H) * 4)};
    for (const Range& r : in)
        if (overlap(rng(o, vb), r)) return SSD_ERR_ALIAS;
    if ((s = pre_launch()) != SSD_OK) return s;
    return from_cuda(launch_gdn_fwd_o(p, q, k, v_new, h, g, o, (cudaStream_t)stream));
}

ssd_status ssd_step(const ssd_dims* d, const void* x, const float* dt, const float* A,
                    const void* B, const void* C, const float* D, float* state, void* y,
                    void* stream) {
    if (!d) return SSD_ERR_NULL;
    ssd_dims dd = *d;
    dd.chunk_size = 64;   // not used by the step; any value passes
    Problem p;
    ssd_status s = make_problem(&dd, &p);
    if (s != SSD_OK) return s;
    if (p.b == 0 || p.L == 0) return SSD_OK;
    if (!x || !dt || !A || !B || !C || !state || !y) return SSD_ERR_NULL;
    if (!aligned16(x) || !aligned16(dt) || !aligned16(A) || !aligned16(B) || !aligned16(C) ||
        !aligned16(D) || !aligned16(state) || !aligned16(y))
        return SSD_ERR_ALIGN;
    const size_t es = (size_t)p.esize;
    const size_t xb = (size_t)(p.b * p.L * p.H * p.P) * es;
    const size_t bcb = (size_t)(p.b * p.L * p.G * p.N) * es;
    const Range in[] = {rng(x, xb), rng(dt, (size_t)(p.b * p.L * p.H) * 4), rng(A, (size_t)p.H * 4),
                        rng(B, bcb), rng(C, bcb), rng(D, (size_t)p.H * 4)};
    const Range sr = rng(state, (size_t)(p.b * p.H * p.P * p.N) * 4), yr = rng(y, xb);
    for (const Range& r : in)
        if (overlap(r, sr) || overlap(r, yr)) return SSD_ERR_ALIAS;
    if (overlap(sr, yr)) return SSD_ERR_ALIAS;
    if ((s = pre_launch()) != SSD_OK) return s;
    return from_cuda(launch_ssd_step(p, x, dt, A, B, C, D, state, y, (cudaStream_t)stream));
}

ssd_status ssd_fwd(const ssd_dims* d, const void* x, const float* dt, const float* A,
                   const void* B, const void* C, const float* D, const float* init_state, void* y,
                   float* final_state, void* workspace, size_t workspace_bytes, void* stream) {
    Problem p;
    ssd_status s = make_problem(d, &p);
    if (s != SSD_OK) return s;
    if (p.b == 0) return SSD_OK;
    if (p.L == 0)  // nothing to compute; the state passes through
        return ssd_fwd_pass_state(d, nullptr, nullptr, nullptr, nullptr, init_state, nullptr,
                                  final_state, nullptr, 0, stream);
    if (!x || !dt || !A || !B || !C || !y) return SSD_ERR_NULL;
    if (!workspace) return SSD_ERR_NULL;
    if (workspace_bytes < ssd_fwd_workspace_bytes(d)) return SSD_ERR_WORKSPACE;
    const size_t es = (size_t)p.esize;
    const size_t xb = (size_t)(p.b * p.L * p.H * p.P) * es;
    const size_t bcb = (size_t)(p.b * p.L * p.G * p.N) * es;
    const size_t sbytes = (size_t)(p.b * p.H * p.P * p.N) * 4;
    if (!aligned16(x) || !aligned16(dt) || !aligned16(A) || !aligned16(B) || !aligned16(C) ||
        !aligned16(D) || !aligned16(init_state) || !aligned16(y) || !aligned16(final_state) ||
        !aligned16(workspace))
        return SSD_ERR_ALIGN;
    const Range in[] = {rng(x, xb), rng(dt, (size_t)(p.b * p.L * p.H) * 4), rng(A, (size_t)p.H * 4),
                        rng(B, bcb), rng(C, bcb), rng(D, (size_t)p.H * 4), rng(init_state, sbytes)};
    const Range ws = rng(workspace, ssd_fwd_workspace_bytes(d));
    const Range yr = rng(y, xb), fr = rng(final_state, sbytes);
    for (int i = 0; i < 7; ++i) {
        if (overlap(in[i], ws) || overlap(in[i], yr)) return SSD_ERR_ALIAS;
        if (i < 6 && overlap(in[i], fr)) return SSD_ERR_ALIAS;
    }
    if (init_state && final_state && init_state != final_state && overlap(in[6], fr))
        return SSD_ERR_ALIAS;
    if (overlap(ws, yr) || overlap(ws, fr) || overlap(yr, fr)) return SSD_ERR_ALIAS;
    if ((s = pre_launch()) != SSD_OK) return s;

    char* w = (char*)workspace;
    float* Gcs = (float*)w;
    float* dtT = (float*)(w + round_up(gcs_bytes(p), kAlign));
    void* hid = (void*)(w + 2 * round_up(gcs_bytes(p), kAlign));
    void* scratch = (void*)(w + 2 * round_up(gcs_bytes(p), kAlign) + round_up(hid_bytes(p), kAlign));
    const bool has_scratch = fwd_pass_state_scratch_bytes(p) > 0;
    unsigned int* ctrl =
        has_scratch ? (unsigned int*)((char*)scratch + fwd_pass_state_ctrl_offset(p)) : nullptr;
    const int ctrl_words = has_scratch ? (int)(fwd_pass_state_ctrl_bytes(p) / 4) : 0;
    cudaStream_t st = (cudaStream_t)stream;
    p.chained = true;
    // chunk_cumsum clears fwd_pass_state's control block on the way
    cudaError_t e = launch_chunk_cumsum(p, dt, A, Gcs, dtT, ctrl, ctrl_words, st);
    if (e == cudaSuccess)
        e = launch_fwd_pass_state(p, x, B, Gcs, dtT, init_state, hid, final_state, scratch, true, st);
    if (e == cudaSuccess) e = launch_compute_out(p, x, B, C, Gcs, dtT, hid, D, y, st);
    return from_cuda(e);
}

}  // extern "C"
