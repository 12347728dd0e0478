// C-ABI of the FGP step library (declarations and contract: include/tvfgp.h).
//
// Host side: argument checks, the FISTA momentum schedule in double, the
// plan of a run (two-step launches that route p and r through the handle's
// two extra dual sets, or one-step launches that ping-pong r with the
// scratch dual), eager launches back to back with no host synchronisation,
// and a CUDA graph of the whole nsteps loop that is re-parameterised in place
// when the buffers, lambda or t0 change (page "TV solver: the FGP step on the
// GPU", sections "Variants" and "What made the difference").  Volumes with
// padded rows run in place on the scalar / 8-byte kernels, or are packed
// into dense buffers for long runs (tvfgp_create_pitched).
#include "tvfgp.h"
#include "fgp_kernels.cuh"
#include "zmarch_tma.cuh"
#include "zmarch2_tma.cuh"
#include "selfcheck.cuh"
#include "cube_tma.cuh"

#include <cuda_runtime.h>

#include <climits>
#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <mutex>
#include <new>
#include <utility>
#include <vector>

using namespace tvfgp;

namespace {

constexpr int kMagic = 0x74766670;   // "tvfp"
constexpr int kVersion = 10000;      // 1.0.0

// launch shapes of the vector kernels (overridable at build time)
#ifndef TVFGP_FUSED_BY
#define TVFGP_FUSED_BY 4
#endif
#ifndef TVFGP_FUSED_ZC
#define TVFGP_FUSED_ZC 8
#endif
constexpr int kFusedBY = TVFGP_FUSED_BY;
constexpr int kFusedZC = TVFGP_FUSED_ZC;
constexpr int kPrimalBY = 8;

// Test hook (tvfgp_debug_fail_allocs): the library's next g_alloc_skip
// device allocations succeed, the g_alloc_fail after them fail.
std::mutex g_alloc_mutex;
int g_alloc_skip = 0, g_alloc_fail = 0;

// Every device allocation of the library goes through here.
template <typename T>
cudaError_t dev_alloc(T **ptr, size_t bytes)
{
    bool fail = false;
    {
        std::lock_guard<std::mutex> lock(g_alloc_mutex);
        if (g_alloc_skip > 0) {
            --g_alloc_skip;
        } else if (g_alloc_fail > 0) {
            --g_alloc_fail;
            fail = true;
        }
    }
    if (fail) {
        *ptr = nullptr;
        return cudaErrorMemoryAllocation;
    }
    return cudaMalloc(reinterpret_cast<void **>(ptr), bytes);
}

// The default vector variant chosen by AUTO.
constexpr int kAutoVariant = TVFGP_VARIANT_ZMARCH2_TMA;

// The parameter struct a kernel takes (checked against the one filled in
// before every launch, so that a kernel id mapped differently by item_cfg
// and fill_item fails instead of launching on the wrong struct).
enum ArgKind { kArgStep, kArgStepH, kArgZmarch, kArgZmarchH, kArgCube, kArgPair, kArgPrimal, kArgDual };

struct LaunchCfg {
    const void *func;
    dim3 grid;
    dim3 block;
    size_t smem;
    int args = kArgStep;
};

// The copy of the final r back from the scratch dual: one contiguous copy of
// `width` bytes, or (pitch != 0, padded rows) `height` rows of `width`
// bytes at a row pitch of `pitch` bytes, leaving the padding untouched.
struct CopySpec {
    size_t width = 0, height = 1, pitch = 0;
};

cudaMemcpy3DParms copy_params(const CopySpec &c, void *dst, const void *src)
{
    cudaMemcpy3DParms q = {};
    q.srcPtr = make_cudaPitchedPtr(const_cast<void *>(src), c.pitch, c.width, c.height);
    q.dstPtr = make_cudaPitchedPtr(dst, c.pitch, c.width, c.height);
    q.extent = make_cudaExtent(c.width, c.height, 1);
    q.kind = cudaMemcpyDeviceToDevice;
    return q;
}

cudaError_t enqueue_copy(const CopySpec &c, void *dst, const void *src, cudaStream_t st)
{
    if (c.pitch == 0) return cudaMemcpyAsync(dst, src, c.width, cudaMemcpyDeviceToDevice, st);
    return cudaMemcpy2DAsync(dst, c.pitch, src, c.pitch, c.width, c.height, cudaMemcpyDeviceToDevice, st);
}

struct GraphEntry {
    int nsteps = -1;
    int variant = -1;
    cudaGraph_t graph = nullptr;
    cudaGraphExec_t exec = nullptr;
    std::vector<cudaGraphNode_t> knodes;
    cudaGraphNode_t cnode = nullptr;
    CopySpec copy;
    // parameters the instantiated graph currently holds
    const float *b = nullptr;
    float *p = nullptr, *r = nullptr;
    float lam = 0.f;
    double t0 = 0.0;
    unsigned long long use = 0;
};

constexpr int kGraphSlots = 4;

}  // namespace

struct tvfgp_handle {
    int magic;
    int nx, ny, nz;
    int px;                        // row pitch of every volume (nx unless created pitched)
    long long N;                   // elements per volume: px*ny*nz
    int variant;
    int graph_on;
    int last_variant;
    long long launches;
    float *scratch;
    float *pair_scratch;        // 9N floats, two-step runs only
    float *zscratch;            // N floats, two-kernel variant only
    int *d_err;
    ZmarchPlan zplan;
    ZmarchPlan zplan_h;            // the z-march over a binary16 dual
    Zmarch2Plan z2plan;
    GraphEntry graphs[kGraphSlots];
    unsigned long long graph_clock;
    // runs on padded rows: a dense handle of the same volume and its
    // staging buffers (b, p, r: 7*nx*ny*nz floats), made on first use
    tvfgp_handle *shadow;
    float *pk;
    int poll_limit;                // bound of the TMA kernels' waits for data (test hook) ...
    int poll_from;                 // ... for the planes of a CTA from this one on
};

namespace {

int from_cuda(cudaError_t e)
{
    if (e == cudaSuccess) return TVFGP_OK;
    return e == cudaErrorMemoryAllocation ? TVFGP_ERR_OOM : TVFGP_ERR_CUDA;
}

bool valid(const tvfgp_handle *h) { return h != nullptr && h->magic == kMagic; }

int check_ptr(const void *p)
{
    if (p == nullptr) return TVFGP_ERR_ARG;
    if (reinterpret_cast<uintptr_t>(p) & 3u) return TVFGP_ERR_ALIGN;
    return TVFGP_OK;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned8(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 7u) == 0; }

// Rows stored without padding: the vector and TMA kernels need it.
bool dense(const tvfgp_handle *h) { return h->px == h->nx; }

// Padded rows the float2 kernel can take: nx and the pitch even.
bool pair_rows(const tvfgp_handle *h) { return !dense(h) && h->nx % 2 == 0 && h->px % 2 == 0; }

// The copy of a whole dual field (3 components) with elements of es bytes:
// contiguous, or only the x < nx part of every padded row.
CopySpec dual_copy(const tvfgp_handle *h, size_t es)
{
    CopySpec c;
    if (dense(h)) {
        c.width = 3 * static_cast<size_t>(h->N) * es;
    } else {
        c.width = static_cast<size_t>(h->nx) * es;
        c.height = 3 * static_cast<size_t>(h->ny) * static_cast<size_t>(h->nz);
        c.pitch = static_cast<size_t>(h->px) * es;
    }
    return c;
}

bool overlap(const void *a, size_t na, const void *b, size_t nb)
{
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return x < y + nb && y < x + na;
}

int check_lambda(float lam)
{
    if (!std::isfinite(lam) || !(lam > 0.0f)) return TVFGP_ERR_ARG;
    const double s = 1.0 / (12.0 * static_cast<double>(lam));
    const float sf = static_cast<float>(s);
    if (!std::isfinite(sf) || !(sf > 0.0f)) return TVFGP_ERR_ARG;
    return TVFGP_OK;
}

// s = 1/(12 lambda), evaluated in double and rounded once to float.
float step_of(float lam) { return static_cast<float>(1.0 / (12.0 * static_cast<double>(lam))); }

// Kernels that are halves of a step of the two-kernel variant.
constexpr int kKernPrimalZVec = 100;     // z = primal of r_src into the handle's z buffer
constexpr int kKernPrimalZScalar = 101;
constexpr int kKernDualZVec = 102;       // the rest of the step, reading that z
constexpr int kKernDualZScalar = 103;
// One-step kernels on a dual stored as binary16.
constexpr int kKernFusedH = 120;
constexpr int kKernScalarH = 121;
constexpr int kKernZmarchH = 122;
// The fused kernel on padded rows (even pitch): on quads moved as two 8-byte
// halves when nx % 4 == 0, on pairs of voxels otherwise.
constexpr int kKernFused2 = 130;
constexpr int kKernFusedP = 131;
constexpr int kFused2BY = 4, kFused2ZC = 8;
// The fused kernel's packing step: padded rows in, dense volumes out (the
// first step of a packed run).
constexpr int kKernPackStep = 132;
// The two-step kernel writing p and r onto padded rows (the last launch of
// a packed run).
constexpr int kKernPairPadded = 133;

// The public variant a kernel belongs to (what tvfgp_last_variant reports).
int public_variant(int kernel)
{
    if (kernel == kKernFused2 || kernel == kKernFusedP || kernel == kKernFusedH || kernel == kKernPackStep)
        return TVFGP_VARIANT_FUSED;
    if (kernel == kKernScalarH) return TVFGP_VARIANT_SCALAR;
    if (kernel == kKernPairPadded) return TVFGP_VARIANT_ZMARCH2_TMA;
    if (kernel == kKernZmarchH) return TVFGP_VARIANT_ZMARCH_TMA;
    if (kernel >= kKernPrimalZVec && kernel <= kKernDualZScalar) return TVFGP_VARIANT_SEPARATE;
    return kernel;
}

// vec_ok: dense rows, nx % 4 == 0 and 16-byte aligned pointers (the float4
// and TMA kernels).  On padded rows every vector variant becomes the float2
// fused kernel when pair_ok (nx and the pitch even, 8-byte aligned pointers),
// else the scalar one; SCALAR and SEPARATE stay.
int resolve_variant(const tvfgp_handle *h, int requested, bool vec_ok, bool pair_ok = false)
{
    int v = requested == TVFGP_VARIANT_AUTO ? kAutoVariant : requested;
    if (!dense(h)) {
        if (v == TVFGP_VARIANT_SCALAR || v == TVFGP_VARIANT_SEPARATE) return v;
        if (!pair_ok) return TVFGP_VARIANT_SCALAR;
        return h->nx % 4 == 0 ? kKernFusedP : kKernFused2;
    }
    if (v == TVFGP_VARIANT_FUSED || v == TVFGP_VARIANT_ZMARCH_TMA || v == TVFGP_VARIANT_ZMARCH2_TMA ||
        v == TVFGP_VARIANT_CUBE_TMA) {
        if (!vec_ok) return TVFGP_VARIANT_SCALAR;
    }
    return v;
}

StepArgs make_args(const tvfgp_handle *h, const float *b, float *p, const float *rs, float *rd,
                   float lam, float m)
{
    StepArgs a;
    a.b = b;
    a.p = p;
    a.rs = rs;
    a.rd = rd;
    a.lam = lam;
    a.s = step_of(lam);
    a.m = m;
    a.nx = h->nx;
    a.ny = h->ny;
    a.nz = h->nz;
    a.N = h->N;
    a.px = h->px;
    return a;
}

// Volumes whose voxel addresses (with one plane of headroom) leave the int
// range run the 64-bit-indexed instances of the fused kernel.
bool wide(const tvfgp_handle *h)
{
    return static_cast<long long>(h->px) * h->ny * (static_cast<long long>(h->nz) + 1) > INT_MAX;
}

template <typename TS, int VW, bool PACK>
const void *fused_kernel(const tvfgp_handle *h)
{
    return wide(h) ? reinterpret_cast<const void *>(&fgp_step_fused4<kFusedBY, kFusedZC, TS, VW, PACK, long long>)
                   : reinterpret_cast<const void *>(&fgp_step_fused4<kFusedBY, kFusedZC, TS, VW, PACK, int>);
}

LaunchCfg step_cfg(const tvfgp_handle *h, int variant)
{
    LaunchCfg c;
    c.smem = 0;
    if (variant == TVFGP_VARIANT_FUSED) {
        c.func = fused_kernel<float, 4, false>(h);
        c.block = dim3(32, kFusedBY, 1);
        c.grid = dim3((h->nx / 4 + 31) / 32, (h->ny + kFusedBY - 1) / kFusedBY,
                      (h->nz + kFusedZC - 1) / kFusedZC);
    } else if (variant == TVFGP_VARIANT_ZMARCH_TMA) {
        c.func = zmarch_kernel();
        c.block = dim3(zmarch_threads(), 1, 1);
        c.grid = zmarch_grid(h->zplan);
        c.smem = zmarch_smem_bytes();
        c.args = kArgZmarch;
    } else if (variant == TVFGP_VARIANT_CUBE_TMA) {
        c.func = cube_kernel();
        c.block = dim3(cube_threads(), 1, 1);
        c.grid = cube_grid(h->nx, h->ny, h->nz);
        c.smem = cube_smem_bytes();
        c.args = kArgCube;
    } else {
        c.func = reinterpret_cast<const void *>(&fgp_step_scalar<float>);
        c.block = dim3(32, 8, 1);
        c.grid = dim3((h->nx + 31) / 32, (h->ny + 7) / 8, h->nz);
    }
    return c;
}


// One kernel launch of a run: a single step (p updated in place, r_src ->
// r_dst), a two-step launch (p_src -> p_dst and r_src -> r_dst), or a half
// of a two-kernel step.
struct Item {
    int kernel;             // a TVFGP_VARIANT_* value
    const float *p_src;
    float *p_dst;
    const float *r_src;
    float *r_dst;
    float m0, m1;           // momentum weights of its step(s)
    // launches of a packed run on padded rows (else left at their defaults):
    const float *b = nullptr;   // this launch's b (nullptr: the run's)
    float *b_out = nullptr;     // packing step: the dense copy of b
    int ipx = 0;                // packing step: the inputs' row pitch ...
    long long in_n = 0;         // ... and elements per volume
    int opx = 0;                // two-step launch: the outputs' row pitch (0: dense) ...
    long long out_n = 0;        // ... and elements per volume
};

// Kernel-argument storage for one launch of any kernel family.
struct KArgs {
    StepArgs a;
    StepArgsT<__half> ah;
    ZmarchArgs za;
    ZmarchArgsT<__half> zah;
    CubeArgs cb;
    Zmarch2Args z2;
    PrimalArgs pa;
    DualArgs da;
    void *ptrs[1];
};

// The member of k that a kernel of ArgKind `kind` takes.
const void *arg_slot(const KArgs &k, int kind)
{
    switch (kind) {
    case kArgStep: return &k.a;
    case kArgStepH: return &k.ah;
    case kArgZmarch: return &k.za;
    case kArgZmarchH: return &k.zah;
    case kArgCube: return &k.cb;
    case kArgPair: return &k.z2;
    case kArgPrimal: return &k.pa;
    case kArgDual: return &k.da;
    }
    return nullptr;
}

LaunchCfg item_cfg(const tvfgp_handle *h, int kernel)
{
    if (kernel == kKernFusedH) {
        LaunchCfg c = step_cfg(h, TVFGP_VARIANT_FUSED);
        c.func = fused_kernel<__half, 4, false>(h);
        c.args = kArgStepH;
        return c;
    }
    if (kernel == kKernScalarH) {
        LaunchCfg c = step_cfg(h, TVFGP_VARIANT_SCALAR);
        c.func = reinterpret_cast<const void *>(&fgp_step_scalar<__half>);
        c.args = kArgStepH;
        return c;
    }
    if (kernel == kKernFusedP) {
        LaunchCfg c = step_cfg(h, TVFGP_VARIANT_FUSED);
        c.func = fused_kernel<float, 2, false>(h);
        return c;
    }
    if (kernel == kKernPackStep) {
        LaunchCfg c = step_cfg(h, TVFGP_VARIANT_FUSED);
        c.func = fused_kernel<float, 2, true>(h);
        return c;
    }
    if (kernel == kKernFused2) {
        LaunchCfg c;
        c.smem = 0;
        c.func = reinterpret_cast<const void *>(&fgp_step_fused2<kFused2BY, kFused2ZC>);
        c.block = dim3(32, kFused2BY, 1);
        c.grid = dim3((h->nx / 2 + 31) / 32, (h->ny + kFused2BY - 1) / kFused2BY,
                      (h->nz + kFused2ZC - 1) / kFused2ZC);
        return c;
    }
    if (kernel == kKernZmarchH) {
        LaunchCfg c;
        c.func = zmarch_kernel<__half>();
        c.block = dim3(zmarch_threads<__half>(), 1, 1);
        c.grid = zmarch_grid(h->zplan_h);
        c.smem = zmarch_smem_bytes<__half>();
        c.args = kArgZmarchH;
        return c;
    }
    if (kernel >= kKernPrimalZVec && kernel <= kKernDualZScalar) {
        LaunchCfg c;
        c.smem = 0;
        c.block = dim3(32, 8, 1);
        c.args = kernel <= kKernPrimalZScalar ? kArgPrimal : kArgDual;
        const bool vec = kernel == kKernPrimalZVec || kernel == kKernDualZVec;
        c.grid = vec ? dim3((h->nx / 4 + 31) / 32, (h->ny + 7) / 8, h->nz)
                     : dim3((h->nx + 31) / 32, (h->ny + 7) / 8, h->nz);
        if (kernel == kKernPrimalZVec) c.func = reinterpret_cast<const void *>(&primal_vec4<8>);
        else if (kernel == kKernPrimalZScalar) c.func = reinterpret_cast<const void *>(&primal_scalar<float>);
        else if (kernel == kKernDualZVec) c.func = reinterpret_cast<const void *>(&dual_from_z_vec4<8>);
        else c.func = reinterpret_cast<const void *>(&dual_from_z_scalar);
        return c;
    }
    if (kernel == TVFGP_VARIANT_ZMARCH2_TMA || kernel == kKernPairPadded) {
        LaunchCfg c;
        c.func = zmarch2_kernel(kernel == kKernPairPadded);
        c.block = dim3(zmarch2_threads(), 1, 1);
        c.grid = h->z2plan.grid;
        c.smem = zmarch2_smem_bytes();
        c.args = kArgPair;
        return c;
    }
    if (kernel != TVFGP_VARIANT_FUSED && kernel != TVFGP_VARIANT_ZMARCH_TMA && kernel != TVFGP_VARIANT_CUBE_TMA &&
        kernel != TVFGP_VARIANT_SCALAR) {
        LaunchCfg c = step_cfg(h, TVFGP_VARIANT_SCALAR);
        c.func = nullptr;                       // unknown kernel id: never launched
        return c;
    }
    return step_cfg(h, kernel);
}

bool fill_item(const tvfgp_handle *h, const Item &it, const float *b_run, float lam, KArgs &k)
{
    const float *b = it.b ? it.b : b_run;
    if (it.kernel == kKernPackStep) {
        // reads (b, p, r) on padded rows, writes dense p', r and b
        k.a = make_args(h, b, const_cast<float *>(it.p_src), it.r_src, it.r_dst, lam, it.m0);
        k.a.px = it.ipx;
        k.a.N = it.in_n;
        k.a.po = it.p_dst;
        k.a.bo = it.b_out;
        k.a.No = h->N;
        k.ptrs[0] = &k.a;
        return it.b_out != nullptr && it.ipx >= h->nx && it.in_n > 0;
    }
    if (it.kernel == kKernFusedH || it.kernel == kKernScalarH || it.kernel == kKernZmarchH) {
        // the dual buffers of a binary16 run travel as float* in an Item
        k.ah.b = b;
        k.ah.p = reinterpret_cast<__half *>(it.p_dst);
        k.ah.rs = reinterpret_cast<const __half *>(it.r_src);
        k.ah.rd = reinterpret_cast<__half *>(it.r_dst);
        k.ah.lam = lam;
        k.ah.s = step_of(lam);
        k.ah.m = it.m0;
        k.ah.nx = h->nx;
        k.ah.ny = h->ny;
        k.ah.nz = h->nz;
        k.ah.N = h->N;
        k.ah.px = h->px;
        if (it.kernel == kKernZmarchH) {
            k.ptrs[0] = &k.zah;
            const bool ok = zmarch_fill(h->zplan_h, k.ah, h->d_err, k.zah);
            k.zah.max_polls = h->poll_limit;
            k.zah.poll_from = h->poll_from;
            return ok;
        }
        k.ptrs[0] = &k.ah;
        return true;
    }
    if (it.kernel == kKernPrimalZVec || it.kernel == kKernPrimalZScalar) {
        k.pa.b = b;
        k.pa.d = it.r_src;
        k.pa.z = h->zscratch;
        k.pa.lam = lam;
        k.pa.nx = h->nx;
        k.pa.ny = h->ny;
        k.pa.nz = h->nz;
        k.pa.N = h->N;
        k.pa.px = h->px;
        k.ptrs[0] = &k.pa;
        return h->zscratch != nullptr;
    }
    if (it.kernel == kKernDualZVec || it.kernel == kKernDualZScalar) {
        k.da.z = h->zscratch;
        k.da.p = it.p_dst;
        k.da.rs = it.r_src;
        k.da.rd = it.r_dst;
        k.da.s = step_of(lam);
        k.da.m = it.m0;
        k.da.nx = h->nx;
        k.da.ny = h->ny;
        k.da.nz = h->nz;
        k.da.N = h->N;
        k.da.px = h->px;
        k.ptrs[0] = &k.da;
        return h->zscratch != nullptr;
    }
    if (it.kernel == TVFGP_VARIANT_ZMARCH2_TMA || it.kernel == kKernPairPadded) {
        k.ptrs[0] = &k.z2;
        const bool ok = zmarch2_fill(h->z2plan, b, it.p_src, it.p_dst, it.r_src, it.r_dst, lam, step_of(lam),
                                     it.m0, it.m1, h->nx, h->ny, h->nz, h->N, h->d_err, k.z2);
        k.z2.max_polls = h->poll_limit;
        k.z2.poll_from = h->poll_from;
        if (it.kernel == TVFGP_VARIANT_ZMARCH2_TMA) return ok;
        k.z2.opx = it.opx;
        k.z2.No = it.out_n;
        return ok && it.opx >= h->nx && it.opx % 2 == 0 && it.out_n > 0;
    }
    k.a = make_args(h, b, it.p_dst, it.r_src, it.r_dst, lam, it.m0);
    if (it.kernel == TVFGP_VARIANT_ZMARCH_TMA) {
        k.ptrs[0] = &k.za;
        const bool ok = zmarch_fill(h->zplan, k.a, h->d_err, k.za);
        k.za.max_polls = h->poll_limit;
        k.za.poll_from = h->poll_from;
        return ok;
    }
    if (it.kernel == TVFGP_VARIANT_CUBE_TMA) {
        k.ptrs[0] = &k.cb;
        const bool ok = cube_fill(k.a, h->d_err, k.cb);
        k.cb.max_polls = h->poll_limit;
        k.cb.poll_from = h->poll_from;
        return ok;
    }
    k.ptrs[0] = &k.a;
    return true;
}

// Buffers a field passes through in `moves` out-of-place updates that start
// and end in buf[0] (moves >= 2): buf[0] -> buf[1] -> buf[2] -> buf[1] ... -> buf[0].
void route(int moves, float *const buf[3], std::vector<float *> &seq)
{
    seq.assign(static_cast<size_t>(moves) + 1, buf[0]);
    if (moves >= 1) seq[1] = buf[1];
    for (int i = 2; i < moves; ++i) seq[i] = seq[i - 1] == buf[1] ? buf[2] : buf[1];
    seq[moves] = buf[0];
}

// The launches of an nsteps run.  Two-step launches are used from four steps
// on; p and r then travel through the handle's two extra buffer sets and end
// in the caller's buffers, with no copy.  Single steps ping-pong r with the
// scratch buffer; an odd count then needs one copy back (*copy_back).
void plan_run(const tvfgp_handle *h, int variant, bool vec_ok, float *p, float *r,
              const std::vector<double> &m, std::vector<Item> &items, bool *copy_back)
{
    const int n = static_cast<int>(m.size());
    items.clear();
    *copy_back = false;
    if (variant == TVFGP_VARIANT_SEPARATE) {
        for (int k = 0; k < n; ++k) {
            const bool even = (k % 2) == 0;
            float *rs = even ? r : h->scratch, *rd = even ? h->scratch : r;
            const float mk = static_cast<float>(m[k]);
            items.push_back({vec_ok ? kKernPrimalZVec : kKernPrimalZScalar, p, p, rs, rd, mk, 0.0f});
            items.push_back({vec_ok ? kKernDualZVec : kKernDualZScalar, p, p, rs, rd, mk, 0.0f});
        }
        *copy_back = (n % 2) == 1;
        return;
    }
    if (variant == TVFGP_VARIANT_ZMARCH2_TMA && n >= 4 && h->pair_scratch != nullptr) {
        const size_t N3 = 3 * static_cast<size_t>(h->N);
        const int pairs = n / 2, single = n % 2;
        float *pb[3] = {p, h->pair_scratch, h->pair_scratch + N3};
        float *rb[3] = {r, h->scratch, h->pair_scratch + 2 * N3};
        std::vector<float *> sp, sr;
        route(pairs, pb, sp);
        route(pairs + single, rb, sr);
        for (int j = 0; j < pairs; ++j)
            items.push_back({TVFGP_VARIANT_ZMARCH2_TMA, sp[j], sp[j + 1], sr[j], sr[j + 1],
                             static_cast<float>(m[2 * j]), static_cast<float>(m[2 * j + 1])});
        if (single)
            items.push_back({TVFGP_VARIANT_ZMARCH_TMA, p, p, sr[pairs], sr[pairs + 1],
                             static_cast<float>(m[n - 1]), 0.0f});
        return;
    }
    const int v = variant == TVFGP_VARIANT_ZMARCH2_TMA ? TVFGP_VARIANT_ZMARCH_TMA : variant;
    for (int k = 0; k < n; ++k) {
        const bool even = (k % 2) == 0;
        items.push_back({v, p, p, even ? r : h->scratch, even ? h->scratch : r,
                         static_cast<float>(m[k]), 0.0f});
    }
    *copy_back = (n % 2) == 1;
}

int launch_item(tvfgp_handle *h, const Item &it, const float *b, float lam, cudaStream_t st)
{
    const LaunchCfg c = item_cfg(h, it.kernel);
    KArgs k;
    if (!fill_item(h, it, b, lam, k) || c.func == nullptr || k.ptrs[0] != arg_slot(k, c.args))
        return TVFGP_ERR_CUDA;
    cudaError_t e = cudaLaunchKernel(c.func, c.grid, c.block, k.ptrs, c.smem, st);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return from_cuda(e);
    }
    h->launches += 1;
    h->last_variant = public_variant(it.kernel);
    return TVFGP_OK;
}

int launch_step(tvfgp_handle *h, int variant, const StepArgs &a, cudaStream_t st)
{
    const Item it{variant, a.p, a.p, a.rs, a.rd, a.m, 0.0f};
    return launch_item(h, it, a.b, a.lam, st);
}

void destroy_graph(GraphEntry &g)
{
    if (g.exec) cudaGraphExecDestroy(g.exec);
    if (g.graph) cudaGraphDestroy(g.graph);
    g = GraphEntry();
}

bool node_params(tvfgp_handle *h, const Item &it, const float *b, float lam, KArgs &ka,
                 cudaKernelNodeParams &kp)
{
    const LaunchCfg c = item_cfg(h, it.kernel);
    const bool ok = fill_item(h, it, b, lam, ka) && c.func != nullptr && ka.ptrs[0] == arg_slot(ka, c.args);
    kp.func = const_cast<void *>(c.func);
    kp.gridDim = c.grid;
    kp.blockDim = c.block;
    kp.sharedMemBytes = static_cast<unsigned>(c.smem);
    kp.kernelParams = ka.ptrs;
    kp.extra = nullptr;
    return ok;
}

int build_graph(tvfgp_handle *h, GraphEntry &g, int variant, const float *b, float *p, float *r,
                float lam, int nsteps, double t0, const std::vector<Item> &items, bool copy_back,
                const CopySpec &copy)
{
    destroy_graph(g);
    cudaError_t e = cudaGraphCreate(&g.graph, 0);
    if (e != cudaSuccess) return from_cuda(e);
    cudaGraphNode_t prev = nullptr;
    g.knodes.resize(items.size());
    for (size_t k = 0; k < items.size(); ++k) {
        KArgs ka;
        cudaKernelNodeParams kp;
        if (!node_params(h, items[k], b, lam, ka, kp)) {
            e = cudaErrorInvalidValue;
            break;
        }
        e = cudaGraphAddKernelNode(&g.knodes[k], g.graph, prev ? &prev : nullptr, prev ? 1 : 0, &kp);
        if (e != cudaSuccess) break;
        prev = g.knodes[k];
    }
    if (e == cudaSuccess && copy_back) {
        if (copy.pitch == 0) {
            e = cudaGraphAddMemcpyNode1D(&g.cnode, g.graph, &prev, 1, r, h->scratch, copy.width,
                                         cudaMemcpyDeviceToDevice);
        } else {
            const cudaMemcpy3DParms q = copy_params(copy, r, h->scratch);
            e = cudaGraphAddMemcpyNode(&g.cnode, g.graph, &prev, 1, &q);
        }
    }
    if (e == cudaSuccess) e = cudaGraphInstantiate(&g.exec, g.graph, 0);
    if (e != cudaSuccess) {
        cudaGetLastError();
        destroy_graph(g);
        return from_cuda(e);
    }
    g.nsteps = nsteps;
    g.variant = variant;
    g.copy = copy;
    g.b = b;
    g.p = p;
    g.r = r;
    g.lam = lam;
    g.t0 = t0;
    return TVFGP_OK;
}

int update_graph(tvfgp_handle *h, GraphEntry &g, const float *b, float *p, float *r, float lam,
                 double t0, const std::vector<Item> &items)
{
    cudaError_t e = cudaSuccess;
    for (size_t k = 0; k < items.size() && e == cudaSuccess; ++k) {
        KArgs ka;
        cudaKernelNodeParams kp;
        if (!node_params(h, items[k], b, lam, ka, kp)) {
            e = cudaErrorInvalidValue;
            break;
        }
        e = cudaGraphExecKernelNodeSetParams(g.exec, g.knodes[k], &kp);
    }
    if (e == cudaSuccess && g.cnode) {
        if (g.copy.pitch == 0) {
            e = cudaGraphExecMemcpyNodeSetParams1D(g.exec, g.cnode, r, h->scratch, g.copy.width,
                                                   cudaMemcpyDeviceToDevice);
        } else {
            const cudaMemcpy3DParms q = copy_params(g.copy, r, h->scratch);
            e = cudaGraphExecMemcpyNodeSetParams(g.exec, g.cnode, &q);
        }
    }
    if (e != cudaSuccess) {
        cudaGetLastError();
        return from_cuda(e);
    }
    g.b = b;
    g.p = p;
    g.r = r;
    g.lam = lam;
    g.t0 = t0;
    return TVFGP_OK;
}

int run_graph(tvfgp_handle *h, int variant, const float *b, float *p, float *r, float lam,
              int nsteps, double t0, const std::vector<Item> &items, bool copy_back,
              const CopySpec &copy, cudaStream_t st)
{
    GraphEntry *g = nullptr;
    for (auto &e : h->graphs)
        if (e.exec && e.nsteps == nsteps && e.variant == variant) g = &e;
    int rc = TVFGP_OK;
    if (g == nullptr) {
        GraphEntry *victim = &h->graphs[0];
        for (auto &e : h->graphs)
            if (!e.exec || e.use < victim->use) victim = &e;
        g = victim;
        rc = build_graph(h, *g, variant, b, p, r, lam, nsteps, t0, items, copy_back, copy);
    } else if (g->b != b || g->p != p || g->r != r || g->lam != lam || g->t0 != t0) {
        rc = update_graph(h, *g, b, p, r, lam, t0, items);
    }
    if (rc != TVFGP_OK) return rc;
    g->use = ++h->graph_clock;
    cudaError_t e = cudaGraphLaunch(g->exec, st);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return from_cuda(e);
    }
    h->launches += static_cast<long long>(items.size());
    h->last_variant = public_variant(items.empty() ? variant : items.front().kernel);
    return TVFGP_OK;
}

// The two extra buffer sets of two-step runs (p twice, r once more; the
// handle's scratch is the other r).
// The z volume of the two-kernel variant.
int ensure_z_scratch(tvfgp_handle *h)
{
    if (h->zscratch) return TVFGP_OK;
    cudaError_t e = dev_alloc(&h->zscratch, sizeof(float) * static_cast<size_t>(h->N));
    if (e != cudaSuccess) {
        cudaGetLastError();
        h->zscratch = nullptr;
        return from_cuda(e);
    }
    return TVFGP_OK;
}

int ensure_pair_scratch(tvfgp_handle *h)
{
    if (h->pair_scratch) return TVFGP_OK;
    cudaError_t e = dev_alloc(&h->pair_scratch, sizeof(float) * 9 * static_cast<size_t>(h->N));
    if (e != cudaSuccess) {
        cudaGetLastError();
        h->pair_scratch = nullptr;
        return from_cuda(e);
    }
    return TVFGP_OK;
}

// Runs on padded rows with at least this many steps are packed into dense
// buffers, run by the dense kernels and unpacked (see tvfgp_run).
constexpr int kPackMinSteps = 4;

int ensure_shadow(tvfgp_handle *h)
{
    if (h->shadow) return TVFGP_OK;
    const size_t n = static_cast<size_t>(h->nx) * h->ny * h->nz;
    cudaError_t e = dev_alloc(&h->pk, sizeof(float) * 7 * n);
    if (e != cudaSuccess) {
        cudaGetLastError();
        h->pk = nullptr;
        return from_cuda(e);
    }
    tvfgp_t s = nullptr;
    const int rc = tvfgp_create_ex(h->nx, h->ny, h->nz, TVFGP_VARIANT_AUTO, 0u, &s);
    if (rc != TVFGP_OK) {
        cudaFree(h->pk);
        h->pk = nullptr;
        return rc;
    }
    h->shadow = s;
    return TVFGP_OK;
}

// `rows` rows of nx floats between a padded buffer (pitch px) and a dense
// one: a kernel when nx % 4 == 0 and the pitch is even (8-byte halves of
// quads), else a 2D copy.
cudaError_t repack(tvfgp_handle *h, float *dst, const float *src, size_t rows, bool to_dense, cudaStream_t st)
{
    const int dp = to_dense ? h->nx : h->px, sp = to_dense ? h->px : h->nx;
    if (h->nx % 4 == 0 && h->px % 2 == 0 && aligned8(dst) && aligned8(src) && rows <= 0x7fffffffULL) {
        repack_rows<<<static_cast<unsigned>(rows), 128, 0, st>>>(dst, dp, src, sp, h->nx);
        h->launches += 1;
        return cudaGetLastError();
    }
    const size_t w = sizeof(float) * static_cast<size_t>(h->nx);
    return cudaMemcpy2DAsync(dst, sizeof(float) * dp, src, sizeof(float) * sp, w, rows, cudaMemcpyDeviceToDevice,
                             st);
}

// The launches of a packed run of n >= 2 steps on padded rows, on the dense
// shadow handle sh: the packing step (step 1: padded b, p, r in; dense b, p',
// r out), one single dense step when the rest is odd (so that the run ends
// on a two-step launch), then two-step launches; the last one writes p and r
// back onto the padded rows.  p and r alternate between the packed buffers
// and the shadow's scratch.
void plan_packed(const tvfgp_handle *h, const tvfgp_handle *sh, const float *b, float *p, float *r,
                 const std::vector<double> &m, std::vector<Item> &items)
{
    const int n = static_cast<int>(m.size());
    const size_t v = static_cast<size_t>(sh->N);
    float *db = h->pk, *pa = h->pk + v, *ra = h->pk + 4 * v;
    float *pb = sh->pair_scratch, *rb = sh->scratch;
    items.clear();
    Item first{kKernPackStep, p, pa, r, ra, static_cast<float>(m[0]), 0.0f};
    first.b = b;
    first.b_out = db;
    first.ipx = h->px;
    first.in_n = h->N;
    items.push_back(first);
    float *cp = pa, *cr = ra, *op = pb, *orr = rb;
    int k = 1;
    if ((n - 1) % 2 == 1) {
        Item one{TVFGP_VARIANT_ZMARCH_TMA, cp, cp, cr, orr, static_cast<float>(m[1]), 0.0f};
        one.b = db;
        items.push_back(one);
        std::swap(cr, orr);
        k = 2;
    }
    for (; k + 1 < n; k += 2) {
        const bool last = k + 2 >= n;
        Item two{last ? kKernPairPadded : TVFGP_VARIANT_ZMARCH2_TMA, cp, last ? p : op, cr, last ? r : orr,
                 static_cast<float>(m[k]), static_cast<float>(m[k + 1])};
        two.b = db;
        if (last) {
            two.opx = h->px;
            two.out_n = h->N;
        }
        items.push_back(two);
        std::swap(cp, op);
        std::swap(cr, orr);
    }
}

// True while `st` is being captured into a CUDA graph.  A run then records
// its launches into the caller's graph one by one (the handle's own graph is
// not replayed inside it) and allocates nothing.
bool capturing(cudaStream_t st)
{
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(st, &cs) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    return cs != cudaStreamCaptureStatusNone;
}

// How a run of nsteps goes on handle h with these buffers: directly on the
// handle's kernels, or through dense buffers (the padded-row runs), either
// with the packing folded into the first step and the unpacking into the
// last two-step launch, or with copies around a dense run.  tma: the TMA
// encoder is available.
enum RunRoute { kRouteDirect = 0, kRoutePackFused = 1, kRoutePackCopy = 2 };

RunRoute run_route(const tvfgp_handle *h, const float *b, const float *p, const float *r, int nsteps, bool tma)
{
    const bool packed_variant = h->variant == TVFGP_VARIANT_AUTO || h->variant == TVFGP_VARIANT_ZMARCH_TMA ||
                                h->variant == TVFGP_VARIANT_ZMARCH2_TMA || h->variant == TVFGP_VARIANT_CUBE_TMA;
    if (dense(h) || h->nx % 4 != 0 || nsteps < kPackMinSteps || !packed_variant) return kRouteDirect;
    if ((h->variant == TVFGP_VARIANT_AUTO || h->variant == TVFGP_VARIANT_ZMARCH2_TMA) && nsteps >= 3 &&
        pair_rows(h) && aligned8(b) && aligned8(p) && aligned8(r) && tma)
        return kRoutePackFused;
    return kRoutePackCopy;
}

}  // namespace

extern "C" {

int tvfgp_version(void) { return kVersion; }

const char *tvfgp_strerror(int code)
{
    switch (code) {
    case TVFGP_OK: return "ok";
    case TVFGP_ERR_ARG: return "invalid argument";
    case TVFGP_ERR_ALIGN: return "pointer not 4-byte aligned";
    case TVFGP_ERR_CUDA: return "CUDA error";
    case TVFGP_ERR_OOM: return "out of memory";
    case TVFGP_ERR_TIMEOUT: return "a bounded device-side wait timed out";
    case TVFGP_ERR_UNSUPPORTED: return "variant not supported for this shape or alignment";
    default: return "unknown status code";
    }
}

int tvfgp_momentum(double t0, int nsteps, double *m, double *t_final)
{
    if (nsteps < 0 || !std::isfinite(t0) || t0 < 1.0) return TVFGP_ERR_ARG;
    double t = t0;
    for (int k = 0; k < nsteps; ++k) {
        const double tn = (1.0 + std::sqrt(1.0 + 4.0 * t * t)) / 2.0;
        if (m) m[k] = (t - 1.0) / tn;
        t = tn;
    }
    if (t_final) *t_final = t;
    return TVFGP_OK;
}

static int create_impl(int nx, int ny, int nz, int px, int variant, unsigned flags, tvfgp_t *out)
{
    if (out == nullptr) return TVFGP_ERR_ARG;
    *out = nullptr;
    if (nx < 1 || ny < 1 || nz < 1 || nx > 65535 || ny > 65535 || nz > 65535) return TVFGP_ERR_ARG;
    if (px < nx || px > 65535) return TVFGP_ERR_ARG;
    if (static_cast<long long>(px) * ny > INT_MAX) return TVFGP_ERR_ARG;     // a plane, in 32 bits
    if (variant < TVFGP_VARIANT_AUTO || variant > TVFGP_VARIANT_CUBE_TMA || flags != 0)
        return TVFGP_ERR_ARG;
    if ((variant == TVFGP_VARIANT_ZMARCH_TMA || variant == TVFGP_VARIANT_ZMARCH2_TMA ||
         variant == TVFGP_VARIANT_CUBE_TMA) &&
        !zmarch_available())
        return TVFGP_ERR_UNSUPPORTED;
    tvfgp_handle *h = new (std::nothrow) tvfgp_handle();
    if (h == nullptr) return TVFGP_ERR_OOM;
    h->magic = kMagic;
    h->nx = nx;
    h->ny = ny;
    h->nz = nz;
    h->px = px;
    h->N = static_cast<long long>(px) * ny * nz;
    h->variant = variant;
    h->graph_on = 0;
    h->last_variant = -1;
    h->launches = 0;
    h->graph_clock = 0;
    h->scratch = nullptr;
    h->pair_scratch = nullptr;
    h->zscratch = nullptr;
    h->d_err = nullptr;
    h->shadow = nullptr;
    h->pk = nullptr;
    h->poll_limit = ZM_MAX_POLLS;
    h->poll_from = 0;
    cudaError_t e = dev_alloc(&h->scratch, sizeof(float) * 3 * static_cast<size_t>(h->N));
    if (e == cudaSuccess) e = dev_alloc(&h->d_err, sizeof(int));
    if (e == cudaSuccess) e = cudaMemset(h->d_err, 0, sizeof(int));
    if (e == cudaSuccess) {
        if (zmarch_plan(nx, ny, nz, &h->zplan) != TVFGP_OK ||
            zmarch_plan<__half>(nx, ny, nz, &h->zplan_h) != TVFGP_OK ||
            zmarch2_plan(nx, ny, nz, &h->z2plan) != TVFGP_OK)
            e = cudaErrorInvalidValue;
    }
    const int want_pairs = variant == TVFGP_VARIANT_ZMARCH2_TMA ||
                           (variant == TVFGP_VARIANT_AUTO && kAutoVariant == TVFGP_VARIANT_ZMARCH2_TMA);
    if (e == cudaSuccess && want_pairs && nx % 4 == 0 && px == nx && ensure_pair_scratch(h) != TVFGP_OK)
        e = cudaErrorMemoryAllocation;
    if (e == cudaSuccess && variant == TVFGP_VARIANT_SEPARATE && ensure_z_scratch(h) != TVFGP_OK)
        e = cudaErrorMemoryAllocation;
    if (e != cudaSuccess) {
        cudaGetLastError();
        cudaFree(h->scratch);
        cudaFree(h->pair_scratch);
        cudaFree(h->zscratch);
        cudaFree(h->d_err);
        h->magic = 0;
        delete h;
        return from_cuda(e);
    }
    *out = h;
    return TVFGP_OK;
}

int tvfgp_create_ex(int nx, int ny, int nz, int variant, unsigned flags, tvfgp_t *out)
{
    return create_impl(nx, ny, nz, nx, variant, flags, out);
}

int tvfgp_create_pitched(int nx, int ny, int nz, int pitch, tvfgp_t *out)
{
    return create_impl(nx, ny, nz, pitch, TVFGP_VARIANT_AUTO, 0u, out);
}

int tvfgp_create(int nx, int ny, int nz, tvfgp_t *out)
{
    return tvfgp_create_ex(nx, ny, nz, TVFGP_VARIANT_AUTO, 0u, out);
}

int tvfgp_destroy(tvfgp_t h)
{
    if (h == nullptr) return TVFGP_OK;
    if (!valid(h)) return TVFGP_ERR_ARG;
    for (auto &g : h->graphs) destroy_graph(g);
    cudaFree(h->scratch);
    cudaFree(h->pair_scratch);
    cudaFree(h->zscratch);
    cudaFree(h->d_err);
    cudaFree(h->pk);
    if (h->shadow) tvfgp_destroy(h->shadow);
    h->magic = 0;
    delete h;
    return TVFGP_OK;
}

int tvfgp_set_variant(tvfgp_t h, int variant)
{
    if (!valid(h) || variant < TVFGP_VARIANT_AUTO || variant > TVFGP_VARIANT_CUBE_TMA)
        return TVFGP_ERR_ARG;
    if (variant == TVFGP_VARIANT_SEPARATE) {
        const int rc = ensure_z_scratch(h);
        if (rc != TVFGP_OK) return rc;
    }
    if ((variant == TVFGP_VARIANT_ZMARCH_TMA || variant == TVFGP_VARIANT_ZMARCH2_TMA ||
         variant == TVFGP_VARIANT_CUBE_TMA) &&
        !zmarch_available())
        return TVFGP_ERR_UNSUPPORTED;
    const int want_pairs = variant == TVFGP_VARIANT_ZMARCH2_TMA ||
                           (variant == TVFGP_VARIANT_AUTO && kAutoVariant == TVFGP_VARIANT_ZMARCH2_TMA);
    if (want_pairs && h->nx % 4 == 0 && dense(h)) {
        const int rc = ensure_pair_scratch(h);
        if (rc != TVFGP_OK) return rc;
    }
    h->variant = variant;
    return TVFGP_OK;
}

int tvfgp_set_graph(tvfgp_t h, int enable)
{
    if (!valid(h)) return TVFGP_ERR_ARG;
    h->graph_on = enable != 0;
    return TVFGP_OK;
}

int tvfgp_last_variant(tvfgp_t h) { return valid(h) ? h->last_variant : -1; }

long long tvfgp_launch_count(tvfgp_t h) { return valid(h) ? h->launches : -1; }

int tvfgp_step(tvfgp_t h, const float *b, float *p, const float *r_src, float *r_dst, float lambda,
               float m, tvfgp_stream_t stream)
{
    if (!valid(h)) return TVFGP_ERR_ARG;
    int rc;
    if ((rc = check_ptr(b)) || (rc = check_ptr(p)) || (rc = check_ptr(r_src)) || (rc = check_ptr(r_dst)))
        return rc;
    if ((rc = check_lambda(lambda))) return rc;
    if (!std::isfinite(m)) return TVFGP_ERR_ARG;
    const size_t v = sizeof(float) * static_cast<size_t>(h->N);
    if (overlap(b, v, p, 3 * v) || overlap(b, v, r_src, 3 * v) || overlap(b, v, r_dst, 3 * v) ||
        overlap(p, 3 * v, r_src, 3 * v) || overlap(p, 3 * v, r_dst, 3 * v) ||
        overlap(r_src, 3 * v, r_dst, 3 * v))
        return TVFGP_ERR_ARG;
    const bool vec_ok = dense(h) && (h->nx % 4 == 0) && aligned16(b) && aligned16(p) && aligned16(r_src) &&
                        aligned16(r_dst);
    const bool pair_ok = pair_rows(h) && aligned8(b) && aligned8(p) && aligned8(r_src) && aligned8(r_dst);
    int variant = resolve_variant(h, h->variant, vec_ok, pair_ok);
    if (variant == TVFGP_VARIANT_ZMARCH2_TMA) variant = TVFGP_VARIANT_ZMARCH_TMA;   // one step only
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (variant == TVFGP_VARIANT_SEPARATE) {
        const Item first{vec_ok ? kKernPrimalZVec : kKernPrimalZScalar, p, p, r_src, r_dst, m, 0.0f};
        const Item second{vec_ok ? kKernDualZVec : kKernDualZScalar, p, p, r_src, r_dst, m, 0.0f};
        int rc2 = launch_item(h, first, b, lambda, st);
        if (rc2 == TVFGP_OK) rc2 = launch_item(h, second, b, lambda, st);
        if (rc2 == TVFGP_OK) h->last_variant = TVFGP_VARIANT_SEPARATE;
        return rc2;
    }
    return launch_step(h, variant, make_args(h, b, p, r_src, r_dst, lambda, m), st);
}

int tvfgp_run(tvfgp_t h, const float *b, float *p, float *r, float lambda, int nsteps, double t0,
              tvfgp_stream_t stream, double *t_final)
{
    if (!valid(h)) return TVFGP_ERR_ARG;
    int rc;
    if ((rc = check_ptr(b)) || (rc = check_ptr(p)) || (rc = check_ptr(r))) return rc;
    if ((rc = check_lambda(lambda))) return rc;
    if (nsteps < 0 || !std::isfinite(t0) || t0 < 1.0) return TVFGP_ERR_ARG;
    const size_t v = sizeof(float) * static_cast<size_t>(h->N);
    if (overlap(b, v, p, 3 * v) || overlap(b, v, r, 3 * v) || overlap(p, 3 * v, r, 3 * v) ||
        overlap(b, v, h->scratch, 3 * v) || overlap(p, 3 * v, h->scratch, 3 * v) ||
        overlap(r, 3 * v, h->scratch, 3 * v))
        return TVFGP_ERR_ARG;
    if (h->pair_scratch && (overlap(b, v, h->pair_scratch, 9 * v) ||
                            overlap(p, 3 * v, h->pair_scratch, 9 * v) ||
                            overlap(r, 3 * v, h->pair_scratch, 9 * v)))
        return TVFGP_ERR_ARG;
    std::vector<double> m(static_cast<size_t>(nsteps));
    double tf = t0;
    tvfgp_momentum(t0, nsteps, m.data(), &tf);
    if (nsteps == 0) {
        if (t_final) *t_final = tf;
        return TVFGP_OK;
    }
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    // Padded rows defeat the 16-byte accesses and the TMA copies of the
    // fastest kernels (a row of 2(nx/2+1) floats is not a multiple of 16
    // bytes), so a run long enough goes through dense buffers.  With the
    // two-step kernel the first step packs and the last launch unpacks; the
    // other TMA variants pack, run and unpack (26 volume moves).  The padding
    // is never written.
    const bool cap = capturing(st);
    const bool use_graph = h->graph_on && !cap;
    const RunRoute route = run_route(h, b, p, r, nsteps, zmarch_available());
    if (route != kRouteDirect && (h->shadow != nullptr || !cap) && ensure_shadow(h) == TVFGP_OK) {
        tvfgp_handle *sh = h->shadow;
        const size_t n = static_cast<size_t>(h->nx) * h->ny * h->nz;
        const size_t rows = static_cast<size_t>(h->ny) * h->nz;
        float *db = h->pk, *dp = h->pk + n, *dr = h->pk + 4 * n;
        // two-step kernel: the packing is fused into the first step and the
        // unpacking into the last launch
        if (route == kRoutePackFused && sh->pair_scratch != nullptr) {
            std::vector<Item> items;
            plan_packed(h, sh, b, p, r, m, items);
            const long long before = sh->launches;
            if (use_graph) {
                rc = run_graph(sh, kKernPackStep, b, p, r, lambda, nsteps, t0, items, false, CopySpec(), st);
            } else {
                for (size_t k = 0; k < items.size() && rc == TVFGP_OK; ++k)
                    rc = launch_item(sh, items[k], db, lambda, st);
            }
            if (rc != TVFGP_OK) return rc;
            h->launches += sh->launches - before;
            h->last_variant = TVFGP_VARIANT_ZMARCH2_TMA;
            if (t_final) *t_final = tf;
            return TVFGP_OK;
        }
        if ((rc = tvfgp_set_variant(sh, h->variant)) || (rc = tvfgp_set_graph(sh, h->graph_on))) return rc;
        cudaError_t e = repack(h, db, b, rows, true, st);
        if (e == cudaSuccess) e = repack(h, dp, p, 3 * rows, true, st);
        if (e == cudaSuccess) e = repack(h, dr, r, 3 * rows, true, st);
        if (e != cudaSuccess) {
            cudaGetLastError();
            return from_cuda(e);
        }
        const long long before = sh->launches;
        rc = tvfgp_run(sh, db, dp, dr, lambda, nsteps, t0, stream, t_final);
        if (rc != TVFGP_OK) return rc;
        h->launches += sh->launches - before;
        e = repack(h, p, dp, 3 * rows, false, st);
        if (e == cudaSuccess) e = repack(h, r, dr, 3 * rows, false, st);
        if (e != cudaSuccess) {
            cudaGetLastError();
            return from_cuda(e);
        }
        h->last_variant = sh->last_variant;
        return TVFGP_OK;
    }
    const bool vec_ok = dense(h) && (h->nx % 4 == 0) && aligned16(b) && aligned16(p) && aligned16(r);
    const bool pair_ok = pair_rows(h) && aligned8(b) && aligned8(p) && aligned8(r);
    const int variant = resolve_variant(h, h->variant, vec_ok, pair_ok);
    std::vector<Item> items;
    bool copy_back = false;
    plan_run(h, variant, vec_ok, p, r, m, items, &copy_back);
    if (use_graph) {
        rc = run_graph(h, variant, b, p, r, lambda, nsteps, t0, items, copy_back, dual_copy(h, 4), st);
    } else {
        for (size_t k = 0; k < items.size() && rc == TVFGP_OK; ++k)
            rc = launch_item(h, items[k], b, lambda, st);
        if (rc == TVFGP_OK && copy_back) {
            cudaError_t e = enqueue_copy(dual_copy(h, 4), r, h->scratch, st);
            if (e != cudaSuccess) {
                cudaGetLastError();
                rc = from_cuda(e);
            }
        }
    }
    if (rc == TVFGP_OK) {
        h->last_variant = public_variant(items.front().kernel);
        if (t_final) *t_final = tf;
    }
    return rc;
}

int tvfgp_primal(tvfgp_t h, const float *b, const float *dual, float lambda, float *z,
                 tvfgp_stream_t stream)
{
    if (!valid(h)) return TVFGP_ERR_ARG;
    int rc;
    if ((rc = check_ptr(b)) || (rc = check_ptr(dual)) || (rc = check_ptr(z))) return rc;
    if ((rc = check_lambda(lambda))) return rc;
    const size_t v = sizeof(float) * static_cast<size_t>(h->N);
    if (overlap(z, v, b, v) || overlap(z, v, dual, 3 * v)) return TVFGP_ERR_ARG;
    PrimalArgs a;
    a.b = b;
    a.d = dual;
    a.z = z;
    a.lam = lambda;
    a.nx = h->nx;
    a.ny = h->ny;
    a.nz = h->nz;
    a.N = h->N;
    a.px = h->px;
    const bool vec_ok = dense(h) && (h->nx % 4 == 0) && aligned16(b) && aligned16(dual) && aligned16(z);
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (vec_ok) {
        dim3 grid((h->nx / 4 + 31) / 32, (h->ny + kPrimalBY - 1) / kPrimalBY, h->nz);
        primal_vec4<kPrimalBY><<<grid, dim3(32, kPrimalBY, 1), 0, st>>>(a);
    } else {
        dim3 grid((h->nx + 31) / 32, (h->ny + 7) / 8, h->nz);
        primal_scalar<float><<<grid, dim3(32, 8, 1), 0, st>>>(a);
    }
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return from_cuda(e);
    h->launches += 1;
    return TVFGP_OK;
}

int tvfgp_run_f16(tvfgp_t h, const float *b, unsigned short *p, unsigned short *r, float lambda,
                  int nsteps, double t0, tvfgp_stream_t stream, double *t_final)
{
    if (!valid(h)) return TVFGP_ERR_ARG;
    int rc;
    if ((rc = check_ptr(b))) return rc;
    if (p == nullptr || r == nullptr) return TVFGP_ERR_ARG;
    if ((reinterpret_cast<uintptr_t>(p) | reinterpret_cast<uintptr_t>(r)) & 1u) return TVFGP_ERR_ALIGN;
    if ((rc = check_lambda(lambda))) return rc;
    if (nsteps < 0 || !std::isfinite(t0) || t0 < 1.0) return TVFGP_ERR_ARG;
    const size_t v = sizeof(float) * static_cast<size_t>(h->N);
    const size_t d = sizeof(unsigned short) * 3 * static_cast<size_t>(h->N);
    if (overlap(b, v, p, d) || overlap(b, v, r, d) || overlap(p, d, r, d) ||
        overlap(b, v, h->scratch, 3 * v) || overlap(p, d, h->scratch, 3 * v) ||
        overlap(r, d, h->scratch, 3 * v))
        return TVFGP_ERR_ARG;
    std::vector<double> m(static_cast<size_t>(nsteps));
    double tf = t0;
    tvfgp_momentum(t0, nsteps, m.data(), &tf);
    if (nsteps == 0) {
        if (t_final) *t_final = tf;
        return TVFGP_OK;
    }
    const bool vec_ok = dense(h) && (h->nx % 4 == 0) && aligned16(b) && (reinterpret_cast<uintptr_t>(p) & 7u) == 0 &&
                        (reinterpret_cast<uintptr_t>(r) & 7u) == 0;
    // The z-march moves rows of whole 16-byte units: nx % 8 == 0 and every
    // component's base 16-byte aligned (N is then a multiple of 8).
    const bool march_ok = dense(h) && zmarch_supported<__half>(h->nx, h->ny, h->nz) && zmarch_available() &&
                          aligned16(b) && aligned16(p) && aligned16(r);
    int kern = kKernScalarH, ran = TVFGP_VARIANT_SCALAR;
    if (h->variant != TVFGP_VARIANT_SCALAR && h->variant != TVFGP_VARIANT_FUSED && march_ok) {
        kern = kKernZmarchH;
        ran = TVFGP_VARIANT_ZMARCH_TMA;
    } else if (h->variant != TVFGP_VARIANT_SCALAR && vec_ok) {
        kern = kKernFusedH;
        ran = TVFGP_VARIANT_FUSED;
    }
    float *pf = reinterpret_cast<float *>(p), *rf = reinterpret_cast<float *>(r);
    std::vector<Item> items;
    for (int k = 0; k < nsteps; ++k) {
        const bool even = (k % 2) == 0;
        items.push_back({kern, pf, pf, even ? rf : h->scratch, even ? h->scratch : rf,
                         static_cast<float>(m[k]), 0.0f});
    }
    const bool copy_back = (nsteps % 2) == 1;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (h->graph_on && !capturing(st)) {
        rc = run_graph(h, kern, b, pf, rf, lambda, nsteps, t0, items, copy_back, dual_copy(h, 2), st);
    } else {
        for (size_t k = 0; k < items.size() && rc == TVFGP_OK; ++k)
            rc = launch_item(h, items[k], b, lambda, st);
        if (rc == TVFGP_OK && copy_back) {
            cudaError_t e = enqueue_copy(dual_copy(h, 2), r, h->scratch, st);
            if (e != cudaSuccess) {
                cudaGetLastError();
                rc = from_cuda(e);
            }
        }
    }
    if (rc == TVFGP_OK) {
        h->last_variant = ran;
        if (t_final) *t_final = tf;
    }
    return rc;
}

int tvfgp_primal_f16(tvfgp_t h, const float *b, const unsigned short *dual, float lambda, float *z,
                     tvfgp_stream_t stream)
{
    if (!valid(h)) return TVFGP_ERR_ARG;
    int rc;
    if ((rc = check_ptr(b)) || (rc = check_ptr(z))) return rc;
    if (dual == nullptr) return TVFGP_ERR_ARG;
    if (reinterpret_cast<uintptr_t>(dual) & 1u) return TVFGP_ERR_ALIGN;
    if ((rc = check_lambda(lambda))) return rc;
    const size_t v = sizeof(float) * static_cast<size_t>(h->N);
    if (overlap(z, v, b, v) || overlap(z, v, dual, sizeof(unsigned short) * 3 * static_cast<size_t>(h->N)))
        return TVFGP_ERR_ARG;
    PrimalArgsT<__half> a;
    a.b = b;
    a.d = reinterpret_cast<const __half *>(dual);
    a.z = z;
    a.lam = lambda;
    a.nx = h->nx;
    a.ny = h->ny;
    a.nz = h->nz;
    a.N = h->N;
    a.px = h->px;
    const bool vec_ok = dense(h) && (h->nx % 4 == 0) && aligned16(b) && aligned16(z) &&
                        (reinterpret_cast<uintptr_t>(dual) & 7u) == 0;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (vec_ok) {
        dim3 grid((h->nx / 4 + 31) / 32, (h->ny + kPrimalBY - 1) / kPrimalBY, h->nz);
        primal_vec4<kPrimalBY, __half><<<grid, dim3(32, kPrimalBY, 1), 0, st>>>(a);
    } else {
        dim3 grid((h->nx + 31) / 32, (h->ny + 7) / 8, h->nz);
        primal_scalar<__half><<<grid, dim3(32, 8, 1), 0, st>>>(a);
    }
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return from_cuda(e);
    h->launches += 1;
    return TVFGP_OK;
}

int tvfgp_check(tvfgp_t h, tvfgp_stream_t stream)
{
    if (!valid(h)) return TVFGP_ERR_ARG;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return from_cuda(e);
    }
    int flag = 0;
    e = cudaMemcpy(&flag, h->d_err, sizeof(int), cudaMemcpyDeviceToHost);
    if (e == cudaSuccess && flag != 0) e = cudaMemset(h->d_err, 0, sizeof(int));
    if (e != cudaSuccess) {
        cudaGetLastError();
        return from_cuda(e);
    }
    if (h->shadow) {                          // kernels of a packed run report there
        const int rc = tvfgp_check(h->shadow, stream);
        if (rc != TVFGP_OK) return rc;
    }
    return flag != 0 ? TVFGP_ERR_TIMEOUT : TVFGP_OK;
}

int tvfgp_host_alloc(size_t bytes, int write_combined, void **out)
{
    if (out == nullptr) return TVFGP_ERR_ARG;
    *out = nullptr;
    if (bytes == 0) return TVFGP_ERR_ARG;
    const unsigned flags = write_combined ? cudaHostAllocWriteCombined : cudaHostAllocDefault;
    const cudaError_t e = cudaHostAlloc(out, bytes, flags);
    if (e != cudaSuccess) {
        cudaGetLastError();
        *out = nullptr;
        return from_cuda(e);
    }
    return TVFGP_OK;
}

int tvfgp_host_free(void *p)
{
    if (p == nullptr) return TVFGP_OK;
    const cudaError_t e = cudaFreeHost(p);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return from_cuda(e);
    }
    return TVFGP_OK;
}

int tvfgp_debug_projection_check(int mode, unsigned long long count, unsigned long long seed,
                                 unsigned long long *out, tvfgp_stream_t stream)
{
    if (mode < 0 || mode > 3 || out == nullptr || (reinterpret_cast<uintptr_t>(out) & 7u)) return TVFGP_ERR_ARG;
    if (mode == 0) count = kNnEnd - kNnFirst;
    else if (count > (1ull << 40)) return TVFGP_ERR_ARG;
    if (count == 0) return TVFGP_OK;
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return from_cuda(e);
    projection_check<<<sms * 8, 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(mode, count, seed, out);
    e = cudaGetLastError();
    return e == cudaSuccess ? TVFGP_OK : from_cuda(e);
}

int tvfgp_debug_set_poll_limit(tvfgp_t h, int polls, int from_plane)
{
    if (!valid(h) || polls > ZM_MAX_POLLS || from_plane < 0) return TVFGP_ERR_ARG;
    const int lim = polls < 0 ? ZM_MAX_POLLS : polls;
    for (tvfgp_handle *x = h; x != nullptr; x = x->shadow) {
        x->poll_limit = lim;
        x->poll_from = polls < 0 ? 0 : from_plane;
        for (auto &g : x->graphs) destroy_graph(g);       // rebuilt with the new limit on next use
    }
    return TVFGP_OK;
}

int tvfgp_debug_fail_allocs(int skip, int count)
{
    if (skip < 0 || count < 0) return TVFGP_ERR_ARG;
    std::lock_guard<std::mutex> lock(g_alloc_mutex);
    g_alloc_skip = count > 0 ? skip : 0;
    g_alloc_fail = count;
    return TVFGP_OK;
}

int tvfgp_debug_plan(int nx, int ny, int nz, int pitch, int variant, int nsteps, double t0, int *route,
                     int *copy_back, int *items, float *m_out, int cap, int *count)
{
    const int px = pitch == 0 ? nx : pitch;
    if (nx < 1 || ny < 1 || nz < 1 || nx > 65535 || ny > 65535 || nz > 65535 || px < nx || px > 65535 ||
        static_cast<long long>(px) * ny > INT_MAX)
        return TVFGP_ERR_ARG;
    if (variant < TVFGP_VARIANT_AUTO || variant > TVFGP_VARIANT_CUBE_TMA || nsteps < 0 || !std::isfinite(t0) ||
        t0 < 1.0 || cap < 0 || route == nullptr || copy_back == nullptr || count == nullptr ||
        (cap > 0 && (items == nullptr || m_out == nullptr)))
        return TVFGP_ERR_ARG;
    // Handles that are never used for CUDA: their buffers are distinct
    // addresses that name the roles, never dereferenced.
    auto fake = [](int role) { return reinterpret_cast<float *>(static_cast<uintptr_t>(role + 1) << 56); };
    const long long nd = static_cast<long long>(nx) * ny * nz;
    tvfgp_handle h{}, sh{};
    h.nx = sh.nx = nx;
    h.ny = sh.ny = ny;
    h.nz = sh.nz = nz;
    h.px = px;
    sh.px = nx;
    h.N = static_cast<long long>(px) * ny * nz;
    sh.N = nd;
    h.variant = variant;
    sh.variant = variant;
    const bool want_pairs = variant == TVFGP_VARIANT_ZMARCH2_TMA ||
                            (variant == TVFGP_VARIANT_AUTO && kAutoVariant == TVFGP_VARIANT_ZMARCH2_TMA);
    h.scratch = fake(3);
    h.pair_scratch = want_pairs && nx % 4 == 0 && px == nx ? fake(4) : nullptr;
    h.pk = fake(7);
    sh.scratch = fake(10);
    sh.pair_scratch = nx % 4 == 0 ? fake(11) : nullptr;
    float *b = fake(0), *p = fake(1), *r = fake(2);
    std::vector<double> m(static_cast<size_t>(nsteps));
    tvfgp_momentum(t0, nsteps, m.data(), nullptr);
    std::vector<Item> plan;
    bool cb = false;
    const RunRoute rt = nsteps == 0 ? kRouteDirect : run_route(&h, b, p, r, nsteps, true);
    if (nsteps == 0) {
    } else if (rt == kRoutePackFused) {
        plan_packed(&h, &sh, b, p, r, m, plan);
    } else if (rt == kRoutePackCopy) {
        float *dp = h.pk + nd, *dr = h.pk + 4 * nd;
        const int v = resolve_variant(&sh, sh.variant, nx % 4 == 0, false);
        plan_run(&sh, v, nx % 4 == 0, dp, dr, m, plan, &cb);
    } else {
        const bool vec_ok = dense(&h) && nx % 4 == 0;
        const int v = resolve_variant(&h, h.variant, vec_ok, pair_rows(&h));
        plan_run(&h, v, vec_ok, p, r, m, plan, &cb);
    }
    // roles: 0 b, 1 p, 2 r (the caller's), 3 scratch dual, 4..6 the pair
    // scratch's three dual sets, 7..9 packed b, p, r, 10 the dense handle's
    // scratch dual, 11..13 its pair scratch's dual sets
    const float *base[14] = {b, p, r, h.scratch, fake(4), fake(4) + 3 * h.N, fake(4) + 6 * h.N, h.pk, h.pk + nd,
                             h.pk + 4 * nd, sh.scratch, fake(11), fake(11) + 3 * nd, fake(11) + 6 * nd};
    auto role = [&](const float *q) {
        if (q == nullptr) return -1;
        for (int k = 0; k < 14; ++k)
            if (q == base[k]) return k;
        return -2;
    };
    *route = static_cast<int>(rt);
    *copy_back = cb ? 1 : 0;
    *count = static_cast<int>(plan.size());
    for (size_t k = 0; k < plan.size() && static_cast<int>(k) < cap; ++k) {
        const Item &it = plan[k];
        int *o = items + 7 * k;
        o[0] = public_variant(it.kernel);
        o[1] = it.b ? role(it.b) : (rt == kRoutePackCopy ? 7 : 0);
        o[2] = role(it.p_src);
        o[3] = role(it.p_dst);
        o[4] = role(it.r_src);
        o[5] = role(it.r_dst);
        o[6] = (it.kernel == TVFGP_VARIANT_ZMARCH2_TMA || it.kernel == kKernPairPadded ? 1 : 0) |
               (it.kernel == kKernPackStep ? 2 : 0) | (it.kernel == kKernPairPadded ? 4 : 0) |
               (it.kernel >= kKernPrimalZVec && it.kernel <= kKernDualZScalar ? 8 : 0);
        m_out[2 * k] = it.m0;
        m_out[2 * k + 1] = it.m1;
    }
    return TVFGP_OK;
}

int tvfgp_debug_chunks(int nx, int ny, int nz, int slots, int *zc, int *z0, int *ze, int cap, int *count)
{
    if (nx < 1 || ny < 1 || nz < 1 || nx > 65535 || ny > 65535 || nz > 65535 || slots < 1 || zc == nullptr ||
        count == nullptr || cap < 0 || (cap > 0 && (z0 == nullptr || ze == nullptr)))
        return TVFGP_ERR_ARG;
    Zmarch2Plan plan{};
    const int tx = (nx + Z2_TX - 1) / Z2_TX, ty = (ny + Z2_TY - 1) / Z2_TY;
    plan.zc = zmarch_pick_zc(tx * ty, nz, slots, TVFGP_Z2_ZC_MAX, TVFGP_Z2_WAVES);
    plan.grid = dim3(tx, ty, (nz + plan.zc - 1) / plan.zc);
    zmarch2_chunks(nz, static_cast<long long>(tx) * ty, slots, &plan);
    *zc = plan.zc;
    *count = static_cast<int>(plan.grid.z);
    // the output planes [z0, ze) of blockIdx.z = j, by the kernel's expressions
    for (int j = 0; j < *count && j < cap; ++j) {
        const int zbase = j < plan.nbig ? 0 : plan.nbig * plan.zc;
        z0[j] = j < plan.nbig ? j * plan.zc : zbase + plan.tap[j - plan.nbig];
        ze[j] = std::min(j < plan.nbig ? z0[j] + plan.zc : zbase + plan.tap[j - plan.nbig + 1], nz);
    }
    return TVFGP_OK;
}

int tvfgp_debug_timeout_probe(tvfgp_t h, int spins, tvfgp_stream_t stream)
{
    if (!valid(h) || spins < 1 || spins > (1 << 24)) return TVFGP_ERR_ARG;
    timeout_probe<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(h->d_err, spins);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return from_cuda(e);
    h->launches += 1;
    return TVFGP_OK;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// tvfgp_run_noalloc: FGP steps with no allocation at all
// ---------------------------------------------------------------------------
//
// For callers that are not allowed to allocate device memory (see the
// header).  The second r buffer of the ping-pong lives in this fixed,
// file-scope device array instead of in a handle: it exists on every GPU
// that loads the library, from module load until the process exits, and is
// shared by every call on that GPU.

static __device__ __align__(256) float g_noalloc_r[3 * static_cast<size_t>(TVFGP_NOALLOC_MAX_VOXELS)];

namespace {

// Device address of g_noalloc_r.  The name g_noalloc_r is only a host-side
// stand-in in host code, never an address a kernel may be given.  Outside
// stream capture the address is looked up on every call, with the calling
// device current, and remembered per device together with the unique id of
// the CUDA context it belongs to.  Under capture the lookup (which may load
// the module) is not made: the remembered address is used only if it was
// taken in the context that is current now, else the call is refused.  So a
// reset device or another context never gets a stale address.
constexpr int kNoallocMaxDevices = 64;
struct NoallocSlot {
    float *addr = nullptr;
    unsigned long long ctx_id = 0;
    bool valid = false;
};
NoallocSlot g_noalloc_slot[kNoallocMaxDevices];
std::mutex g_noalloc_mu;

// Unique id of the current CUDA context (ids are never reused within a
// process), from the driver's cuCtxGetCurrent and cuCtxGetId.
bool current_context_id(unsigned long long *id)
{
    static const auto fns = [] {
        void *get = nullptr, *gid = nullptr;
        cudaDriverEntryPointQueryResult q1, q2;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &get, 12000, cudaEnableDefault, &q1) !=
                cudaSuccess || q1 != cudaDriverEntryPointSuccess)
            get = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &gid, 12000, cudaEnableDefault, &q2) !=
                cudaSuccess || q2 != cudaDriverEntryPointSuccess)
            gid = nullptr;
        cudaGetLastError();
        return std::make_pair(reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(get),
                              reinterpret_cast<PFN_cuCtxGetId_v12000>(gid));
    }();
    if (fns.first == nullptr || fns.second == nullptr) return false;
    CUcontext ctx = nullptr;
    if (fns.first(&ctx) != CUDA_SUCCESS || ctx == nullptr) return false;
    return fns.second(ctx, id) == CUDA_SUCCESS;
}

int noalloc_scratch(cudaStream_t st, float **out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kNoallocMaxDevices) {
        cudaGetLastError();
        return TVFGP_ERR_CUDA;
    }
    const bool cap = capturing(st);
    unsigned long long id = 0;
    const bool have_id = current_context_id(&id);
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    NoallocSlot &slot = g_noalloc_slot[dev];
    if (cap) {
        if (!slot.valid || !have_id || slot.ctx_id != id) return TVFGP_ERR_ARG;
        *out = slot.addr;
        return TVFGP_OK;
    }
    void *p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_r);
    if (e != cudaSuccess || p == nullptr) {
        cudaGetLastError();
        return TVFGP_ERR_CUDA;
    }
    slot.addr = static_cast<float *>(p);
    slot.ctx_id = id;
    slot.valid = have_id;
    *out = slot.addr;
    return TVFGP_OK;
}

}  // namespace

extern "C" int tvfgp_debug_noalloc_scratch(void **addr, unsigned long long *bytes)
{
    if (addr == nullptr || bytes == nullptr) return TVFGP_ERR_ARG;
    float *p = nullptr;
    const int rc = noalloc_scratch(nullptr, &p);
    if (rc) return rc;
    *addr = p;
    *bytes = sizeof(g_noalloc_r);
    return TVFGP_OK;
}

extern "C" int tvfgp_run_noalloc(int nx, int ny, int nz, const float *b, float *p, float *r,
                                 float lambda, int nsteps, double t0, tvfgp_stream_t stream,
                                 double *t_final)
{
    if (nx < 1 || ny < 1 || nz < 1 || nx > 65535 || ny > 65535 || nz > 65535) return TVFGP_ERR_ARG;
    const long long N = static_cast<long long>(nx) * ny * nz;
    if (N > TVFGP_NOALLOC_MAX_VOXELS) return TVFGP_ERR_UNSUPPORTED;
    int rc;
    if ((rc = check_ptr(b)) || (rc = check_ptr(p)) || (rc = check_ptr(r))) return rc;
    if ((rc = check_lambda(lambda))) return rc;
    if (nsteps < 0 || !std::isfinite(t0) || t0 < 1.0) return TVFGP_ERR_ARG;
    const size_t v = sizeof(float) * static_cast<size_t>(N);
    if (overlap(b, v, p, 3 * v) || overlap(b, v, r, 3 * v) || overlap(p, 3 * v, r, 3 * v))
        return TVFGP_ERR_ARG;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    float *scratch = nullptr;
    if ((rc = noalloc_scratch(st, &scratch))) return rc;
    // a caller buffer anywhere in the array would be overwritten by some call
    const size_t whole = sizeof(g_noalloc_r);
    if (overlap(b, v, scratch, whole) || overlap(p, 3 * v, scratch, whole) || overlap(r, 3 * v, scratch, whole))
        return TVFGP_ERR_ARG;

    // Same launches as tvfgp_run's eager path, with the momentum schedule
    // evaluated step by step (no host buffer either).
    const bool vec_ok = (nx % 4 == 0) && aligned16(b) && aligned16(p) && aligned16(r);
    StepArgs a;
    a.b = b;
    a.p = p;
    a.lam = lambda;
    a.s = step_of(lambda);
    a.nx = nx;
    a.ny = ny;
    a.nz = nz;
    a.N = N;
    a.px = nx;
    dim3 grid, block;
    const void *fn;
    if (vec_ok) {
        fn = reinterpret_cast<const void *>(&fgp_step_fused4<kFusedBY, kFusedZC>);
        block = dim3(32, kFusedBY, 1);
        grid = dim3((nx / 4 + 31) / 32, (ny + kFusedBY - 1) / kFusedBY, (nz + kFusedZC - 1) / kFusedZC);
    } else {
        fn = reinterpret_cast<const void *>(&fgp_step_scalar<float>);
        block = dim3(32, 8, 1);
        grid = dim3((nx + 31) / 32, (ny + 7) / 8, nz);
    }
    double t = t0;
    for (int k = 0; k < nsteps; ++k) {
        const double tn = (1.0 + std::sqrt(1.0 + 4.0 * t * t)) / 2.0;
        a.m = static_cast<float>((t - 1.0) / tn);
        t = tn;
        const bool even = (k % 2) == 0;
        a.rs = even ? r : scratch;
        a.rd = even ? scratch : r;
        void *args[] = {&a};
        const cudaError_t e = cudaLaunchKernel(fn, grid, block, args, 0, st);
        if (e != cudaSuccess) {
            cudaGetLastError();
            return from_cuda(e);
        }
    }
    if (nsteps % 2 == 1) {
        const cudaError_t e = cudaMemcpyAsync(r, scratch, 3 * v, cudaMemcpyDeviceToDevice, st);
        if (e != cudaSuccess) {
            cudaGetLastError();
            return from_cuda(e);
        }
    }
    if (t_final) *t_final = t;
    return TVFGP_OK;
}
