// ssd_host.cu -- ssd_fwd on host buffers.  The batch is cut into contiguous
// slices; each slice's inputs are copied in on one stream, its forward pass
// runs on the caller's stream, and its outputs are copied out on a third, so
// that the host-device traffic of one slice overlaps the computation (and the
// traffic in the other direction) of the others.  Batch elements are
// independent recurrences, so a slice is an ssd_fwd problem of its own.
// include/ssd.h states the contract.
#include <vector>

#include "ssd_internal.cuh"

namespace {

constexpr size_t kAlign = 256;
constexpr int kMaxSlices = 64;

size_t up(size_t v) { return (v + kAlign - 1) / kAlign * kAlign; }

// Bytes per batch element of each tensor.
struct PerBatch {
    size_t x, dt, bc, st;   // x (and y); dt; B (and C); a state (init_state, final_state)
};
PerBatch per_batch(const ssd_dims* d) {
    const size_t es = d->dtype == SSD_BF16 ? 2 : 4;
    return {(size_t)(d->seqlen * d->nheads * d->headdim) * es, (size_t)(d->seqlen * d->nheads) * 4,
            (size_t)(d->seqlen * d->ngroups * d->dstate) * es,
            (size_t)(d->nheads * d->headdim * d->dstate) * 4};
}

// One staging slot: the device copies of a slice's inputs and outputs and its
// ssd_fwd workspace, each 256-byte aligned; offsets from the slot's start.
struct Slot {
    size_t x, dt, B, C, init, y, fin, ws, ws_bytes, bytes;
};
Slot slot_layout(const ssd_dims* d, int64_t bs) {
    const PerBatch z = per_batch(d);
    ssd_dims ds = *d;
    ds.batch = bs;
    Slot s;
    size_t o = 0;
    s.x = o;    o += up(z.x * bs);
    s.dt = o;   o += up(z.dt * bs);
    s.B = o;    o += up(z.bc * bs);
    s.C = o;    o += up(z.bc * bs);
    s.init = o; o += up(z.st * bs);
    s.y = o;    o += up(z.x * bs);
    s.fin = o;  o += up(z.st * bs);
    s.ws = o;
    s.ws_bytes = up(ssd_fwd_workspace_bytes(&ds));
    o += s.ws_bytes;
    s.bytes = o;
    return s;
}

struct Plan {
    int64_t bs, ns;   // batch elements per slice, number of (non-empty) slices
    int nslots;
};
Plan plan(const ssd_dims* d, int nslices) {
    Plan p;
    p.bs = (d->batch + nslices - 1) / nslices;
    p.ns = (d->batch + p.bs - 1) / p.bs;
    p.nslots = p.ns > 1 ? 2 : 1;
    return p;
}

struct HRange {
    uintptr_t lo, hi;
};
HRange hr(const void* p, size_t n) { return {(uintptr_t)p, (uintptr_t)p + n}; }
bool hoverlap(HRange a, HRange b) {
    return a.lo != 0 && b.lo != 0 && a.hi > a.lo && b.hi > b.lo && a.lo < b.hi && b.lo < a.hi;
}

}  // namespace

extern "C" size_t ssd_fwd_host_staging_bytes(const ssd_dims* d, int nslices) {
    size_t g = 0, h = 0;
    if (!d || ssd_intermediate_bytes(d, &g, &h) != SSD_OK) return 0;
    if (d->batch == 0 || nslices < 1 || nslices > kMaxSlices || nslices > d->batch) return 0;
    const Plan p = plan(d, nslices);
    return 2 * up((size_t)d->nheads * 4) + (size_t)p.nslots * slot_layout(d, p.bs).bytes;
}

extern "C" ssd_status ssd_fwd_host(const ssd_dims* d, const void* x, const float* dt,
                                   const float* A, const void* B, const void* C, const float* D,
                                   const float* init_state, void* y, float* final_state,
                                   void* staging, size_t staging_bytes, int nslices,
                                   void* const* streams) {
    if (!d) return SSD_ERR_NULL;
    size_t g = 0, h = 0;
    ssd_status s = ssd_intermediate_bytes(d, &g, &h);
    if (s != SSD_OK) return s;
    if (d->batch == 0) return SSD_OK;
    if (nslices < 1 || nslices > kMaxSlices || nslices > d->batch) return SSD_ERR_SHAPE;
    if (!streams || !A) return SSD_ERR_NULL;
    if (d->seqlen > 0 && (!x || !dt || !B || !C || !y)) return SSD_ERR_NULL;
    if (!staging) return SSD_ERR_NULL;
    if (((uintptr_t)staging & (kAlign - 1)) != 0) return SSD_ERR_ALIGN;
    if (staging_bytes < ssd_fwd_host_staging_bytes(d, nslices)) return SSD_ERR_WORKSPACE;
    const PerBatch z = per_batch(d);
    const int64_t b = d->batch;
    {   // outputs must not overlap inputs (host ranges)
        // (final_state may be init_state itself: each slice's state is copied in
        // before its result is copied out over it)
        const HRange in[] = {hr(x, z.x * b), hr(dt, z.dt * b), hr(A, (size_t)d->nheads * 4),
                             hr(B, z.bc * b), hr(C, z.bc * b), hr(D, D ? (size_t)d->nheads * 4 : 0),
                             hr(init_state, init_state ? z.st * b : 0)};
        const HRange yr = hr(y, z.x * b), fr = hr(final_state, final_state ? z.st * b : 0);
        for (int i = 0; i < 7; ++i) {
            if (hoverlap(in[i], yr)) return SSD_ERR_ALIAS;
            if (hoverlap(in[i], fr) && !(i == 6 && init_state == final_state)) return SSD_ERR_ALIAS;
        }
        if (hoverlap(yr, fr)) return SSD_ERR_ALIAS;
    }
    {   // a bounded wait of an earlier launch gave up: report it, enqueue nothing
        const ssd_status t = ssd::timeout_pending();
        if (t != SSD_OK) return t;
    }

    const Plan p = plan(d, nslices);
    char* base = (char*)staging;
    float* dA = (float*)base;
    float* dD = (float*)(base + up((size_t)d->nheads * 4));
    char* slots = base + 2 * up((size_t)d->nheads * 4);
    const Slot L = slot_layout(d, p.bs);
    cudaStream_t sc = (cudaStream_t)streams[0], si = (cudaStream_t)streams[1],
                 so = (cudaStream_t)streams[2];

    // events: two for the error path, entry, then per slice inputs-in,
    // computed, outputs-out
    std::vector<cudaEvent_t> ev;
    const size_t nev = 3 + 3 * (size_t)p.ns;
    ev.reserve(nev);
    auto done = [&](ssd_status r) {
        if (r != SSD_OK && ev.size() == nev) {
            // whatever was enqueued finishes before the caller's stream moves on
            cudaEventRecord(ev[0], si);
            cudaEventRecord(ev[1], so);
            cudaStreamWaitEvent(sc, ev[0], 0);
            cudaStreamWaitEvent(sc, ev[1], 0);
            cudaGetLastError();
        }
        for (cudaEvent_t e : ev) cudaEventDestroy(e);   // released once they complete
        return r;
    };
    for (size_t i = 0; i < nev; ++i) {
        cudaEvent_t e;
        if (cudaEventCreateWithFlags(&e, cudaEventDisableTiming) != cudaSuccess) {
            cudaGetLastError();
            return done(SSD_ERR_CUDA);
        }
        ev.push_back(e);
    }
    cudaEvent_t entry = ev[2];
    auto in_ready = [&](int64_t k) { return ev[3 + 3 * k]; };
    auto computed = [&](int64_t k) { return ev[4 + 3 * k]; };
    auto out_done = [&](int64_t k) { return ev[5 + 3 * k]; };
    auto ok = [](cudaError_t e) { return e == cudaSuccess; };
    auto h2d = [&](void* dst, const void* src, size_t n) {
        return n == 0 || ok(cudaMemcpyAsync(dst, src, n, cudaMemcpyHostToDevice, si));
    };
    auto d2h = [&](void* dst, const void* src, size_t n) {
        return n == 0 || ok(cudaMemcpyAsync(dst, src, n, cudaMemcpyDeviceToHost, so));
    };

    // the copies start after the work the caller enqueued on its stream
    bool good = ok(cudaEventRecord(entry, sc)) && ok(cudaStreamWaitEvent(si, entry, 0)) &&
                ok(cudaStreamWaitEvent(so, entry, 0)) && h2d(dA, A, (size_t)d->nheads * 4) &&
                (D == nullptr || h2d(dD, D, (size_t)d->nheads * 4));
    for (int64_t k = 0; good && k < p.ns; ++k) {
        const int64_t b0 = k * p.bs, bk = (b - b0 < p.bs) ? b - b0 : p.bs;
        char* t = slots + (size_t)(k % p.nslots) * L.bytes;   // this slice's slot
        // inputs of slice k, once slice k - nslots (same slot) has been computed
        good = (k < p.nslots || ok(cudaStreamWaitEvent(si, computed(k - p.nslots), 0))) &&
               h2d(t + L.x, (const char*)x + b0 * z.x, bk * z.x) &&
               h2d(t + L.dt, (const char*)dt + b0 * z.dt, bk * z.dt) &&
               h2d(t + L.B, (const char*)B + b0 * z.bc, bk * z.bc) &&
               h2d(t + L.C, (const char*)C + b0 * z.bc, bk * z.bc) &&
               (init_state == nullptr ||
                h2d(t + L.init, (const char*)init_state + b0 * z.st, bk * z.st)) &&
               ok(cudaEventRecord(in_ready(k), si));
        if (!good) break;
        // the forward pass of slice k, once its inputs are in and slice
        // k - nslots's outputs are out
        good = ok(cudaStreamWaitEvent(sc, in_ready(k), 0)) &&
               (k < p.nslots || ok(cudaStreamWaitEvent(sc, out_done(k - p.nslots), 0)));
        if (!good) break;
        ssd_dims dk = *d;
        dk.batch = bk;
        s = ssd_fwd(&dk, t + L.x, (const float*)(t + L.dt), dA, t + L.B, t + L.C,
                    D ? dD : nullptr, init_state ? (const float*)(t + L.init) : nullptr, t + L.y,
                    final_state ? (float*)(t + L.fin) : nullptr, t + L.ws, L.ws_bytes, sc);
        if (s != SSD_OK) return done(s);
        // outputs of slice k
        good = ok(cudaEventRecord(computed(k), sc)) && ok(cudaStreamWaitEvent(so, computed(k), 0)) &&
               d2h((char*)y + b0 * z.x, t + L.y, bk * z.x) &&
               (final_state == nullptr ||
                d2h((char*)final_state + b0 * z.st, t + L.fin, bk * z.st)) &&
               ok(cudaEventRecord(out_done(k), so));
    }
    // the caller's stream reaches the end of the call once the last copy is out
    good = good && ok(cudaStreamWaitEvent(sc, out_done(p.ns - 1), 0));
    if (!good) {
        cudaGetLastError();
        return done(SSD_ERR_CUDA);
    }
    return done(SSD_OK);
}
