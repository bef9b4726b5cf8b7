// zero_step.cu -- the host side of the ZeRO update step on one GB300 (sm_103a):
// plans and their argument checks, launch shapes and the split of long ranges
// into chained sub-launches, the workspace layout, and the C entry points that
// include/zero_gb300.h declares.  The kernels and the step's arithmetic are in
// zero_kernels.cuh.

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <map>
#include <mutex>
#include <tuple>
#include <utility>

#include "zero_common.cuh"
#include "zero_elem.cuh"
#include "zero_gb300.h"
#include "zero_kernels.cuh"

namespace {

// ------------------------------------------------------------------ host side

using StepKernel = void (*)(StepArgs);

template <int NT, bool B>
struct FusedK {
    static constexpr StepKernel fn = zero_fused_kernel<NT, B, false>;
};
template <int NT, bool B>
struct FusedAccK {
    static constexpr StepKernel fn = zero_fused_kernel<NT, B, true>;
};
template <int NT, bool B>
struct ReduceK {
    static constexpr StepKernel fn = zero_reduce_kernel<NT, B>;
};

template <int NT, bool B>
struct StagedK {
    static constexpr StepKernel fn = zero_fused_staged_kernel<NT, B>;
};
template <int NT, bool B>
struct AccumK {
    static constexpr StepKernel fn = zero_accum_kernel<NT, B>;
};

// The rank count a kernel instance is compiled for: N itself for 1, 2, 4 and
// 8, else 0 (the instance that reads N at run time).
int compiled_ranks(int N) { return (N == 1 || N == 2 || N == 4 || N == 8) ? N : 0; }

template <template <int, bool> class K>
StepKernel pick(int N, bool bf16) {
    switch (compiled_ranks(N)) {
        case 1: return bf16 ? K<1, true>::fn : K<1, false>::fn;
        case 2: return bf16 ? K<2, true>::fn : K<2, false>::fn;
        case 4: return bf16 ? K<4, true>::fn : K<4, false>::fn;
        case 8: return bf16 ? K<8, true>::fn : K<8, false>::fn;
        default: return bf16 ? K<0, true>::fn : K<0, false>::fn;
    }
}


// Launch shape of a step kernel: the register kernels take one 8-element group
// per thread and no dynamic shared memory; the staged kernel one tile of
// `tile` elements per CTA and `smem` bytes of stages.
struct Shape {
    int threads = kThreads;
    size_t smem = 0;
    int tile = 0;  // 0: not tiled
};

// Persistent grid: as many CTAs as fit on the device at once (a multiple of
// the SM count), fewer if the range is small.
// The grid of a launch with work for every resident CTA: every SM full, at
// most kMaxGrid CTAs.
int full_grid(const void* fn, int device, const Shape& sh = Shape{}) {
    const int64_t full =
        static_cast<int64_t>(sm_count(device)) * resident_ctas(fn, device, sh.threads, sh.smem);
    return full > kMaxGrid ? kMaxGrid : (full < 1 ? 1 : static_cast<int>(full));
}

int grid_for(const void* fn, int device, int64_t n8, const Shape& sh = Shape{}) {
    const int64_t need = sh.tile > 0 ? (n8 * kVec + sh.tile - 1) / sh.tile
                                     : (n8 + sh.threads - 1) / sh.threads;
    const int full = full_grid(fn, device, sh);
    return need < 1 ? 1 : (need < full ? static_cast<int>(need) : full);
}

// Launches fn over a.n8 groups.  With overlap_previous the launch may begin
// while the kernel before it on the stream drains (programmatic dependent
// launch); only first-pass bucket launches of one step, whose elements are
// disjoint from the previous bucket's, ask for it.
bool launch(StepKernel fn, int device, const StepArgs& a, cudaStream_t stream,
            bool overlap_previous = false, const Shape& sh = Shape{}) {
    const int grid = grid_for(reinterpret_cast<const void*>(fn), device, a.n8, sh);
    if (overlap_previous || sh.smem > 0) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(static_cast<unsigned>(grid));
        cfg.blockDim = dim3(static_cast<unsigned>(sh.threads));
        cfg.dynamicSmemBytes = sh.smem;
        cfg.stream = stream;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = overlap_previous ? 1 : 0;
        if (cudaLaunchKernelEx(&cfg, fn, a) != cudaSuccess) return false;
    } else {
        fn<<<grid, kThreads, 0, stream>>>(a);
    }
    g_launches.fetch_add(1, std::memory_order_relaxed);
    return cudaGetLastError() == cudaSuccess;
}

// Largest range one launch covers.  A longer range (a large bucket, or the
// whole vector when the step has one bucket) is split into near-equal
// sub-launches chained by programmatic dependent launch: each one starts
// streaming while the previous drains.  Measured on flat vectors of 1.2e8 to
// 3e9 elements, a cap of 4M elements per launch was the most consistent
// choice, against 6M to 16M.  For Psi = 1e9, N = 8 in 25M buckets it gave
// 6.76 TB/s, against 6.54 TB/s with one launch per bucket.
constexpr int64_t kLaunchElems = int64_t(1) << 22;
constexpr int64_t kLaunchAlignGroups = 32;  // 256 elements

// Launches fn over elements [begin, end) of a (a multiple of kVec long), in
// sub-launches of at most kLaunchElems.  The first sub-launch overlaps the
// kernel before it on the stream only if overlap_first; the others always
// follow a sub-launch of the same range.
// Where the first-pass launches of a step put their norm partials: rows of
// their own while the workspace has rows left (see finish_cta), then the
// shared slots.  rows == nullptr or capacity 0: the shared slots only.
struct RowSource {
    double* rows = nullptr;      // capacity rows of kMaxGrid slots
    double* carry = nullptr;
    int32_t capacity = 0;
    int32_t* used = nullptr;     // rows handed out so far in this step
    int32_t* width = nullptr;    // the slots of the latest row that count
    int32_t* shared = nullptr;   // set to 1 once a launch adds to the shared slots
    int32_t mode_without_row = kSharedSlot;
};

bool launch_range(StepKernel fn, int device, StepArgs a, int64_t begin, int64_t end,
                  cudaStream_t stream, bool overlap_first, const Shape& sh = Shape{},
                  int64_t overrun_groups = 0, RowSource* rs = nullptr) {
    const int64_t groups = (end - begin) / kVec;
    if (groups <= 0) return true;
    const int64_t parts = (groups * kVec + kLaunchElems - 1) / kLaunchElems;
    // Sub-launch sizes are a multiple of kLaunchAlignGroups, so each sub-launch
    // starts as aligned as the range does.  With a range starting on a
    // 512-byte boundary, every warp's 16-byte-per-lane access then covers
    // whole 128-byte lines.  Split at an odd offset instead, each warp access
    // straddles one more line: measured 8-9 % slower.
    int64_t per = (groups + parts - 1) / parts;
    per = (per + kLaunchAlignGroups - 1) / kLaunchAlignGroups * kLaunchAlignGroups;
    for (int64_t k = 0, g0 = 0; g0 < groups; ++k, g0 += per) {
        a.begin = begin + g0 * kVec;
        a.n8 = (groups - g0 < per) ? groups - g0 : per;
        if (g0 + per >= groups) a.n8 += overrun_groups;  // the last launch (debug tests only)
        if (rs != nullptr) {
            if (rs->mode_without_row != kNoPartial && *rs->used < rs->capacity) {
                const int32_t j = *rs->used;
                a.partial_mode = kOwnRow;
                a.partials = rs->rows + static_cast<int64_t>(j) * kMaxGrid;
                // as wide as a full launch of this kernel: a shorter launch
                // zeroes the slots past its grid
                a.row_width = full_grid(reinterpret_cast<const void*>(fn), device, sh);
                a.prev_row = j > 0 ? a.partials - kMaxGrid : nullptr;
                a.prev_width = j > 0 ? *rs->width : 0;
                a.carry = rs->carry;
                a.carry_in = j >= 2 ? 1 : 0;
                *rs->width = a.row_width;
                *rs->used = j + 1;
            } else {
                a.partial_mode = rs->mode_without_row;
                if (a.partial_mode == kSharedSlot) *rs->shared = 1;
            }
        }
        if (!launch(fn, device, a, stream, k > 0 || overlap_first, sh)) return false;
    }
    return true;
}


// The staged kernel's TMA copies read device memory only (not pinned host or
// managed memory, which the register kernels can also read).
bool device_memory(const void* ptr) {
    cudaPointerAttributes attr;
    if (cudaPointerGetAttributes(&attr, ptr) != cudaSuccess) {
        cudaGetLastError();  // clear the error that query may leave behind
        return false;
    }
    return attr.type == cudaMemoryTypeDevice;
}

// Stages of the staged kernel for N ranks: as many as fit (at most
// kMaxStages) in kStagedSmemLimit, at least two.  Fills a.stages,
// a.stage_bytes and the launch shape; false if two stages do not fit.
bool staged_shape(StepKernel fn, int device, int N, bool bf16, StepArgs& a, Shape& sh) {
    const int tile = staged_tile(compiled_ranks(N), bf16);  // the instance pick<StagedK> chose
    const size_t stage = static_cast<size_t>(N) * tile * (bf16 ? 2 : 4) + 3 * size_t(tile) * 4;
    int stages = kMaxStages;
    while (stages >= 2 && stages * (stage + 16) > kStagedSmemLimit) --stages;
    if (stages < 2) return false;
    {
        static std::mutex mu;
        static std::map<std::pair<const void*, int>, bool> opted_in;
        std::lock_guard<std::mutex> lock(mu);
        auto key = std::make_pair(reinterpret_cast<const void*>(fn), device);
        if (!opted_in[key]) {
            if (cudaFuncSetAttribute(reinterpret_cast<const void*>(fn),
                                     cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     static_cast<int>(kStagedSmemLimit)) != cudaSuccess)
                return false;
            opted_in[key] = true;
        }
    }
    a.stages = stages;
    a.stage_bytes = static_cast<uint32_t>(stage);
    sh.threads = 32 * (tile / 128) + 32;  // Staged<NT, bf16>::kThreads
    sh.smem = stages * stage + 2 * stages * sizeof(uint64_t);
    sh.tile = tile;
    return true;
}

struct Span {
    uintptr_t lo, hi;
    bool written;
};

bool overlaps(const Span& x, const Span& y) { return x.lo < y.hi && y.lo < x.hi; }

bool disjoint(const Span* s, int n) {
    for (int i = 0; i < n; ++i)
        for (int k = i + 1; k < n; ++k) {
            if (!s[i].written && !s[k].written) continue;  // read-only buffers may share memory
            if (overlaps(s[i], s[k])) return false;
        }
    return true;
}

bool valid_hparams(const zero_adam_hparams* hp) {
    if (hp == nullptr) return false;
    auto finite = [](double x) { return std::isfinite(x); };
    return finite(hp->lr) && hp->lr >= 0.0 && finite(hp->beta1) && hp->beta1 >= 0.0 &&
           hp->beta1 < 1.0 && finite(hp->beta2) && hp->beta2 >= 0.0 && hp->beta2 < 1.0 &&
           finite(hp->eps) && hp->eps > 0.0 && finite(hp->weight_decay) &&
           hp->weight_decay >= 0.0 && finite(hp->max_grad_norm) && hp->max_grad_norm >= 0.0 &&
           hp->step >= 1 && (hp->skip_on_overflow == 0 || hp->skip_on_overflow == 1) &&
           hp->micro_batches >= 0 && hp->bucket_elems >= 0 &&
           hp->bucket_elems % ZERO_BUCKET_ALIGN == 0;
}

int32_t micro_batches_of(const zero_adam_hparams* hp) {
    return hp->micro_batches > 1 ? hp->micro_batches : 1;
}

// The update must wait for the step-wide decision: with clipping, or when a
// skipped in-place step would have nothing left to restore from.
bool needs_two_passes(const zero_adam_hparams* hp, bool in_place) {
    return hp->max_grad_norm > 0.0 || (in_place && hp->skip_on_overflow);
}

Scalars make_scalars(const zero_adam_hparams* hp, int32_t N, float loss_scale) {
    Scalars s;
    const double t = static_cast<double>(hp->step);
    // the batch mean covers N ranks times the micro-batches accumulated
    s.inv = static_cast<float>(1.0 / (static_cast<double>(N) * micro_batches_of(hp) *
                                      static_cast<double>(loss_scale)));
    s.b1 = static_cast<float>(hp->beta1);
    s.omb1 = static_cast<float>(1.0 - hp->beta1);
    s.b2 = static_cast<float>(hp->beta2);
    s.omb2 = static_cast<float>(1.0 - hp->beta2);
    s.eps = static_cast<float>(hp->eps);
    s.step_size = static_cast<float>(hp->lr / (1.0 - std::pow(hp->beta1, t)));
    s.sbc2 = static_cast<float>(std::sqrt(1.0 - std::pow(hp->beta2, t)));
    s.decay = static_cast<float>(1.0 - hp->lr * hp->weight_decay);
    s.use_decay = hp->weight_decay != 0.0 ? 1 : 0;
    return s;
}

// The part of the workspace every step needs: the control block and shared
// slots, plus the FP32 combined gradient when the step keeps one.
size_t workspace_bytes(int64_t psi_pad, const zero_adam_hparams* hp, bool in_place) {
    size_t b = kGradOffset;
    if (needs_two_passes(hp, in_place) || micro_batches_of(hp) > 1)
        b += static_cast<size_t>(psi_pad) * sizeof(float);
    return b;
}

size_t align256(size_t x) { return (x + 255) / 256 * 256; }

// Bytes of a rows area holding `rows` rows: the finalize block sums, then the
// rows.
size_t rows_area_bytes(int64_t rows) {
    if (rows <= 0) return 0;
    return kRowsHeaderBytes + static_cast<size_t>(rows) * kRowBytes;
}

// First-pass launches in one pass over psi_pad elements in buckets of
// hp->bucket_elems (launch_range's split), at most kRowCap.
int64_t launches_per_pass(int64_t psi_pad, const zero_adam_hparams* hp) {
    auto parts = [](int64_t len) -> int64_t {
        const int64_t groups = len / kVec;
        return groups <= 0 ? 0 : (groups * kVec + kLaunchElems - 1) / kLaunchElems;
    };
    if (psi_pad <= 0) return 0;
    const int64_t bucket = hp->bucket_elems > 0 ? hp->bucket_elems : psi_pad;
    const int64_t full = psi_pad / bucket;
    const int64_t total = (full > kRowCap ? kRowCap : full) * parts(bucket) + parts(psi_pad - full * bucket);
    return total > kRowCap ? kRowCap : total;
}

// Rows a rows area of `avail` bytes holds.
int32_t rows_capacity(size_t avail) {
    if (avail <= kRowsHeaderBytes) return 0;
    const int64_t c = static_cast<int64_t>((avail - kRowsHeaderBytes) / kRowBytes);
    return static_cast<int32_t>(c > kRowCap ? kRowCap : c);
}

// The rows area of a plan's workspace.
struct RowArea {
    double* carry = nullptr;
    double* rows = nullptr;
};

RowArea row_area(const zero_plan* p) {
    RowArea r;
    if (p->row_capacity <= 0) return r;
    char* base = static_cast<char*>(p->workspace) + p->rows_offset;
    r.carry = reinterpret_cast<double*>(base);
    r.rows = reinterpret_cast<double*>(base + kRowsHeaderBytes);
    return r;
}

size_t grad_elem_bytes(int32_t dtype) { return dtype == ZERO_GRAD_BF16 ? 2u : 4u; }

// The buffers a step writes, as spans (for the overlap checks).
int written_spans(const zero_plan* p, Span* out) {
    const uintptr_t n = static_cast<uintptr_t>(p->psi_pad);
    int k = 0;
    auto add = [&](const void* ptr, uintptr_t bytes) {
        if (ptr != nullptr)
            out[k++] = Span{reinterpret_cast<uintptr_t>(ptr), reinterpret_cast<uintptr_t>(ptr) + bytes,
                            true};
    };
    add(p->dst_master, 4 * n);
    add(p->dst_m, 4 * n);
    add(p->dst_v, 4 * n);
    add(p->dst_w_bf16, 2 * n);
    // the workspace up to the end of what the step touches (its rows area too)
    const size_t needed = p->grad_accum != nullptr ? kGradOffset
                                                   : workspace_bytes(p->psi_pad, &p->hp, p->in_place != 0);
    const size_t touched = p->row_capacity > 0
                               ? static_cast<size_t>(p->rows_offset) + rows_area_bytes(p->row_capacity)
                               : needed;
    add(p->workspace, touched);
    if (p->grad_accum != nullptr) add(p->grad_accum, 4 * n);
    return k;
}

// Debug builds only, to test the checks: ZERO_DEBUG_TEST_OVERRUN=g makes the
// last launch of each pass over the vector cover g more 8-element groups past
// its end (at most 1024), which the kernels' checks must skip.  The release
// build never overruns.
int64_t debug_test_overrun() {
#ifdef ZERO_DEBUG
    static const int64_t g = [] {
        const char* v = std::getenv("ZERO_DEBUG_TEST_OVERRUN");
        const long long x = v != nullptr ? std::atoll(v) : 0;
        return static_cast<int64_t>(x < 0 ? 0 : (x > 1024 ? 1024 : x));
    }();
    return g;
#else
    return 0;
#endif
}

StepArgs base_args(const zero_plan* p) {
    char* ws = static_cast<char*>(p->workspace);
    StepArgs a{};
    for (int i = 0; i < p->N; ++i) a.grads[i] = p->grads[i];
    a.src_master = p->src_master;
    a.src_m = p->src_m;
    a.src_v = p->src_v;
    a.src_w = p->src_w_bf16;
    a.dst_master = p->dst_master;
    a.dst_m = p->dst_m;
    a.dst_v = p->dst_v;
    a.dst_w = p->dst_w_bf16;
    a.gws = p->grad_accum != nullptr ? p->grad_accum : reinterpret_cast<float*>(ws + kGradOffset);
    a.partials = reinterpret_cast<double*>(ws + kPartialsOffset);
    a.ctrl = reinterpret_cast<Ctrl*>(ws);
    a.s = make_scalars(&p->hp, p->N, p->loss_scale);
    a.sdev = p->policy != nullptr ? &a.ctrl->scalars : nullptr;
    a.N = p->N;
    a.clip = p->hp.max_grad_norm > 0.0 ? 1 : 0;
    a.gbase = 0;
    a.pingpong = p->current_set != nullptr ? 1 : 0;
    a.limit = p->psi_pad;
    a.grad_lo = 0;
    a.grad_hi = p->psi_pad;
    a.partial_mode = kSharedSlot;
    return a;
}

int plan_init(zero_plan* plan, const void* const* grads, int32_t grad_dtype,
              const float* src_master, const float* src_m, const float* src_v,
              const uint16_t* src_w, float* dst_master, float* dst_m, float* dst_v,
              uint16_t* dst_w, int64_t psi_pad, int32_t N, const zero_adam_hparams* hp,
              float loss_scale, void* workspace, size_t workspace_bytes_given,
              bool allow_null_grads, float* grad_accum = nullptr) {
    if (plan == nullptr) return ZERO_ERR_ARG;
    const bool in_place = (dst_master == src_master);
    if (grads == nullptr || N < 1 || N > ZERO_MAX_RANKS || psi_pad < 0 || psi_pad > ZERO_MAX_ELEMS ||
        (grad_dtype != ZERO_GRAD_BF16 && grad_dtype != ZERO_GRAD_FP32) || !valid_hparams(hp) ||
        !(loss_scale > 0.0f) || !std::isfinite(loss_scale))
        return ZERO_ERR_ARG;
    if (psi_pad % (static_cast<int64_t>(N) * ZERO_PAD_UNIT) != 0) return ZERO_ERR_ARG;
    const bool have_data = psi_pad > 0;
    const void* bufs[] = {src_master, src_m, src_v, dst_master, dst_m, dst_v, dst_w};
    for (const void* p : bufs)
        if (have_data && p == nullptr) return ZERO_ERR_ARG;
    if (!in_place && hp->skip_on_overflow && have_data && src_w == nullptr) return ZERO_ERR_ARG;
    if (in_place && (src_m != dst_m || src_v != dst_v)) return ZERO_ERR_ARG;
    for (int i = 0; i < N; ++i) {
        if (have_data && grads[i] == nullptr && !allow_null_grads) return ZERO_ERR_ARG;
        if (!aligned(grads[i], ZERO_ALIGN_BYTES)) return ZERO_ERR_ALIGN;
    }
    for (const void* p : bufs)
        if (!aligned(p, ZERO_ALIGN_BYTES)) return ZERO_ERR_ALIGN;
    if (!aligned(src_w, ZERO_ALIGN_BYTES)) return ZERO_ERR_ALIGN;
    float* accum_dev = nullptr;  // grad_accum as the device addresses it
    if (grad_accum != nullptr) {
        if (!aligned(grad_accum, ZERO_ALIGN_BYTES)) return ZERO_ERR_ALIGN;
        cudaPointerAttributes attr;
        if (cudaPointerGetAttributes(&attr, grad_accum) != cudaSuccess ||
            attr.devicePointer == nullptr) {
            cudaGetLastError();  // clear the error that query may leave behind
            return ZERO_ERR_ARG;
        }
        accum_dev = static_cast<float*>(attr.devicePointer);
    }
    const size_t need = grad_accum != nullptr ? kGradOffset : workspace_bytes(psi_pad, hp, in_place);
    if (workspace == nullptr || workspace_bytes_given < need || !aligned(workspace, 256))
        return ZERO_ERR_WORKSPACE;

    zero_plan p{};
    for (int i = 0; i < N; ++i) p.grads[i] = grads[i];
    p.src_master = src_master;
    p.src_m = src_m;
    p.src_v = src_v;
    p.src_w_bf16 = src_w;
    p.dst_master = dst_master;
    p.dst_m = dst_m;
    p.dst_v = dst_v;
    p.dst_w_bf16 = dst_w;
    p.workspace = workspace;
    p.workspace_bytes = workspace_bytes_given;
    p.psi_pad = psi_pad;
    p.cursor = 0;
    p.hp = *hp;
    p.loss_scale = loss_scale;
    p.grad_dtype = grad_dtype;
    p.N = N;
    p.in_place = in_place ? 1 : 0;
    p.two_pass = (needs_two_passes(hp, in_place) || grad_accum != nullptr) ? 1 : 0;
    p.grad_accum = accum_dev;
    p.state = 1;
    // whatever the workspace holds beyond what the step needs becomes rows of
    // norm partials (see finish_cta)
    p.rows_offset = static_cast<int64_t>(align256(need));
    p.row_capacity = workspace_bytes_given > static_cast<size_t>(p.rows_offset)
                         ? rows_capacity(workspace_bytes_given - static_cast<size_t>(p.rows_offset))
                         : 0;
    p.rows_used = 0;
    p.row_width = 0;
    p.shared_slots_used = 0;

    if (have_data) {
        const uintptr_t n = static_cast<uintptr_t>(psi_pad);
        Span sp[ZERO_MAX_RANKS + 12];  // grads + up to 6 written + 4 read-only
        int k = written_spans(&p, sp);
        auto add = [&](const void* ptr, uintptr_t bytes) {
            if (ptr != nullptr)
                sp[k++] = Span{reinterpret_cast<uintptr_t>(ptr),
                               reinterpret_cast<uintptr_t>(ptr) + bytes, false};
        };
        for (int i = 0; i < N; ++i) add(grads[i], n * grad_elem_bytes(grad_dtype));
        if (!in_place) {
            add(src_master, 4 * n);
            add(src_m, 4 * n);
            add(src_v, 4 * n);
            if (hp->skip_on_overflow) add(src_w, 2 * n);
        }
        if (!disjoint(sp, k)) return ZERO_ERR_OVERLAP;
    }
    *plan = p;
    return ZERO_OK;
}

int plan_begin(zero_plan* p, void* stream) {
    NvtxRange range("zero_plan_begin");
    if (p == nullptr || p->state < 1) return ZERO_ERR_ARG;
    if (cudaMemsetAsync(p->workspace, 0, kGradOffset, static_cast<cudaStream_t>(stream)) !=
        cudaSuccess)
        return ZERO_ERR_CUDA;
    if (p->policy != nullptr || p->current_set != nullptr) {
        // the window of bias corrections travels with the launch, unless the
        // plan reads them from the caller's table
        PolicyTable window{};
        if (p->policy_table == nullptr) {
            zero_adam_hparams hp = p->hp;
            const int32_t n = p->policy_t_count < ZERO_POLICY_WINDOW ? p->policy_t_count
                                                                      : ZERO_POLICY_WINDOW;
            for (int32_t i = 0; i < n; ++i) {
                hp.step = p->policy_t_first + i;
                const Scalars si = make_scalars(&hp, p->N, p->loss_scale);
                window.step_size[i] = si.step_size;
                window.sbc2[i] = si.sbc2;
            }
        }
        const Scalars base = make_scalars(&p->hp, p->N, p->loss_scale);
        zero_step_prologue_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(
            static_cast<const zero_device_policy*>(p->policy),
            reinterpret_cast<Ctrl*>(p->workspace), base, window, p->policy_table,
            p->policy_t_first, p->policy_t_count,
            static_cast<double>(p->N) * micro_batches_of(&p->hp),
            static_cast<const int32_t*>(p->current_set));
        g_launches.fetch_add(1, std::memory_order_relaxed);
        if (cudaGetLastError() != cudaSuccess) return ZERO_ERR_CUDA;
    }
    p->cursor = 0;
    p->micro_batch = 0;
    p->rows_used = 0;
    p->row_width = 0;
    p->shared_slots_used = 0;
    p->state = 2;
    return ZERO_OK;
}

int plan_bucket(zero_plan* p, int64_t begin, int64_t end, const void* const* bucket_grads,
                void* stream) {
    NvtxRange range("zero_plan_bucket");
    if (p == nullptr || p->state != 2) return ZERO_ERR_ARG;
    if (begin != p->cursor || end <= begin || end > p->psi_pad ||
        (end % ZERO_BUCKET_ALIGN != 0 && end != p->psi_pad))
        return ZERO_ERR_ARG;
    StepArgs a = base_args(p);
    if (bucket_grads != nullptr) {
        Span written[6];
        const int nw = written_spans(p, written);
        const uintptr_t bytes = static_cast<uintptr_t>(end - begin) * grad_elem_bytes(p->grad_dtype);
        for (int i = 0; i < p->N; ++i) {
            if (bucket_grads[i] == nullptr) return ZERO_ERR_ARG;
            if (!aligned(bucket_grads[i], ZERO_ALIGN_BYTES)) return ZERO_ERR_ALIGN;
            const Span g{reinterpret_cast<uintptr_t>(bucket_grads[i]),
                         reinterpret_cast<uintptr_t>(bucket_grads[i]) + bytes, false};
            for (int k = 0; k < nw; ++k)
                if (overlaps(g, written[k])) return ZERO_ERR_OVERLAP;
            a.grads[i] = bucket_grads[i];
        }
        a.gbase = begin;
        a.grad_lo = begin;   // a staging slot holds this bucket only
        a.grad_hi = end;
    } else {
        for (int i = 0; i < p->N; ++i)
            if (p->grads[i] == nullptr) return ZERO_ERR_ARG;
    }
    int device = 0;
    if (cudaGetDevice(&device) != cudaSuccess) return ZERO_ERR_CUDA;
    const bool bf16 = p->grad_dtype == ZERO_GRAD_BF16;
    const int32_t k = micro_batches_of(&p->hp);
    if (p->smem_staging < ZERO_STAGING_REGISTERS || p->smem_staging > ZERO_STAGING_TMA_TEST_STALL)
        return ZERO_ERR_ARG;
    StepKernel fn;
    Shape shape;
    if (k == 1 && !p->two_pass && p->smem_staging != ZERO_STAGING_REGISTERS) {
        fn = pick<StagedK>(p->N, bf16);
        if (!staged_shape(fn, device, p->N, bf16, a, shape)) return ZERO_ERR_ARG;
        // the plan's own gradient buffers once per pass (at its first bucket),
        // a bucket's own pointers every time
        if (bucket_grads != nullptr || begin == 0)
            for (int i = 0; i < p->N; ++i)
                if (!device_memory(a.grads[i])) return ZERO_ERR_ARG;
        if (begin == 0 && bucket_grads != nullptr)
            for (int i = 0; i < p->N; ++i)
                if (p->grads[i] != nullptr && !device_memory(p->grads[i])) return ZERO_ERR_ARG;
        if (begin == 0 &&
            (!device_memory(p->src_master) || !device_memory(p->src_m) || !device_memory(p->src_v)))
            return ZERO_ERR_ARG;
        // with ping-pong sets the copies may read either set
        if (begin == 0 && p->current_set != nullptr &&
            (!device_memory(p->dst_master) || !device_memory(p->dst_m) || !device_memory(p->dst_v)))
            return ZERO_ERR_ARG;
        a.test_stall = p->smem_staging == ZERO_STAGING_TMA_TEST_STALL ? 1 : 0;
    } else if (k > 1 && p->micro_batch == k - 1 && !p->two_pass) {
        // the last micro-batch of a step with no second pass: accumulate and
        // update in one pass, without writing the accumulator back
        fn = pick<FusedAccK>(p->N, bf16);
    } else if (k > 1) {
        fn = pick<AccumK>(p->N, bf16);
        a.acc_first = p->micro_batch == 0 ? 1 : 0;
        a.acc_last = p->micro_batch == k - 1 ? 1 : 0;
    } else {
        fn = p->two_pass ? pick<ReduceK>(p->N, bf16) : pick<FusedK>(p->N, bf16);
    }
    // Overlap with the previous bucket only when that launch is the one right
    // before this on the stream.  The caller promises that by setting
    // overlap_buckets (zero_step does).  A bucket read from a staging slot
    // follows the wait for that slot's copy, so that caller leaves the flag at
    // 0.  The first bucket of a pass (begin == 0) never overlaps: when
    // accumulating it reads what the previous micro-batch wrote.
    const bool overlap = p->overlap_buckets != 0 && begin > 0;
    // the launches' norm partials: rows of their own while the workspace has
    // rows left; the accumulate passes before the last micro-batch have none
    const RowArea ra = row_area(p);
    RowSource rs;
    rs.rows = ra.rows;
    rs.carry = ra.carry;
    rs.capacity = p->row_capacity;
    rs.used = &p->rows_used;
    rs.width = &p->row_width;
    rs.shared = &p->shared_slots_used;
    rs.mode_without_row = (k > 1 && p->micro_batch < k - 1) ? kNoPartial : kSharedSlot;
    if (!launch_range(fn, device, a, begin, end, static_cast<cudaStream_t>(stream), overlap, shape,
                      end == p->psi_pad ? debug_test_overrun() : 0, &rs))
        return ZERO_ERR_CUDA;
    p->cursor = end;
    // accumulating: a micro-batch that covered the vector hands over to the
    // next, whose first bucket starts at 0 again.  That first bucket is never
    // overlapped (begin == 0), because it reads what this micro-batch wrote.
    if (p->cursor == p->psi_pad && p->micro_batch < k - 1) {
        p->micro_batch += 1;
        p->cursor = 0;
    }
    return ZERO_OK;
}

int plan_end(zero_plan* p, zero_step_result* result, void* stream_handle) {
    NvtxRange range("zero_plan_end");
    if (p == nullptr || p->state != 2 || p->cursor != p->psi_pad ||
        p->micro_batch != micro_batches_of(&p->hp) - 1)
        return ZERO_ERR_ARG;
    zero_step_result* result_dev = nullptr;
    if (result != nullptr) {
        cudaPointerAttributes attr;
        if (cudaPointerGetAttributes(&attr, result) != cudaSuccess || attr.devicePointer == nullptr) {
            cudaGetLastError();  // clear the error that query may leave behind
            return ZERO_ERR_ARG;
        }
        result_dev = static_cast<zero_step_result*>(attr.devicePointer);
    }
    int device = 0;
    if (cudaGetDevice(&device) != cudaSuccess) return ZERO_ERR_CUDA;
    cudaStream_t stream = static_cast<cudaStream_t>(stream_handle);
    StepArgs a = base_args(p);
    Ctrl* ctrl = a.ctrl;
    if (result_dev == nullptr) result_dev = &ctrl->result;

    {
        // A programmatic dependent of whatever kernel precedes it on the stream
        // (normally the last bucket's last launch); it waits for that grid to
        // complete before it reads anything.
        const RowArea ra = row_area(p);
        const int32_t n_rows = p->rows_used;
        const double* last_row = n_rows > 0 ? ra.rows + static_cast<int64_t>(n_rows - 1) * kMaxGrid
                                            : nullptr;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(1);
        cfg.blockDim = dim3(kFinalizeThreads);
        cfg.stream = stream;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        if (cudaLaunchKernelEx(&cfg, zero_finalize_kernel, ctrl, static_cast<const double*>(a.partials),
                               p->shared_slots_used, last_row, n_rows > 0 ? p->row_width : 0,
                               static_cast<const double*>(n_rows >= 2 ? ra.carry : nullptr),
                               p->hp.max_grad_norm, static_cast<int>(p->hp.skip_on_overflow),
                               result_dev, static_cast<zero_device_policy*>(p->policy),
                               static_cast<int32_t*>(p->current_set)) != cudaSuccess)
            return ZERO_ERR_CUDA;
    }
    g_launches.fetch_add(1, std::memory_order_relaxed);
    if (cudaGetLastError() != cudaSuccess) return ZERO_ERR_CUDA;

    if (p->two_pass) {
        // the first update launch waits for the finalize kernel in stream order
        if (!launch_range(zero_update_kernel, device, a, 0, p->psi_pad, stream, false, Shape{},
                          debug_test_overrun()))
            return ZERO_ERR_CUDA;
    } else if (!p->in_place && p->current_set == nullptr &&
               (p->hp.skip_on_overflow || p->policy != nullptr ||
                p->smem_staging != ZERO_STAGING_REGISTERS || kDebugBuild)) {
        // a skipped step (overflow, a t outside the policy's window, a timed-out
        // staged wait, or in a debug build an access the checks skipped) must
        // leave dst equal to src.  With ping-pong sets the current set stays
        // current instead, and nothing is copied.
        a.begin = 0;
        a.n8 = p->psi_pad / kVec + debug_test_overrun();
        if (!launch(zero_restore_kernel, device, a, stream)) return ZERO_ERR_CUDA;
    }
    p->state = 1;

    if (result == nullptr) {
        zero_step_result host;
        if (cudaMemcpyAsync(&host, &ctrl->result, sizeof host, cudaMemcpyDeviceToHost, stream) !=
                cudaSuccess ||
            cudaStreamSynchronize(stream) != cudaSuccess)
            return ZERO_ERR_CUDA;
        return host.status;
    }
    return ZERO_OK;
}

// zero_step and zero_step_into: one plan, walked bucket by bucket.
int run_step(const void* const* grads, int32_t grad_dtype, const float* src_master,
             const float* src_m, const float* src_v, const uint16_t* src_w, float* dst_master,
             float* dst_m, float* dst_v, uint16_t* dst_w, int64_t psi_pad, int32_t N,
             const zero_adam_hparams* hp, float loss_scale, void* workspace,
             size_t workspace_bytes_given, zero_step_result* result, void* stream) {
    NvtxRange range("zero_step");
    if (hp != nullptr && micro_batches_of(hp) > 1) return ZERO_ERR_ARG;  // one batch only
    zero_plan plan;
    int rc = plan_init(&plan, grads, grad_dtype, src_master, src_m, src_v, src_w, dst_master, dst_m,
                       dst_v, dst_w, psi_pad, N, hp, loss_scale, workspace, workspace_bytes_given,
                       false);
    if (rc != ZERO_OK) return rc;
    plan.overlap_buckets = 1;  // the buckets below are launched back to back
    if ((rc = plan_begin(&plan, stream)) != ZERO_OK) return rc;
    const int64_t bucket = hp->bucket_elems > 0 ? hp->bucket_elems : psi_pad;
    for (int64_t b0 = 0; b0 < psi_pad; b0 += bucket) {
        const int64_t b1 = (psi_pad - b0 > bucket) ? b0 + bucket : psi_pad;
        if ((rc = plan_bucket(&plan, b0, b1, nullptr, stream)) != ZERO_OK) return rc;
    }
    return plan_end(&plan, result, stream);
}

}  // namespace

extern "C" size_t zero_workspace_bytes(int64_t psi_pad, const zero_adam_hparams* hp,
                                       int32_t in_place) {
    if (psi_pad < 0 || psi_pad > ZERO_MAX_ELEMS || hp == nullptr) return 0;
    return align256(workspace_bytes(psi_pad, hp, in_place != 0)) +
           rows_area_bytes(launches_per_pass(psi_pad, hp));
}

extern "C" int zero_step(const void* const* grads, int32_t grad_dtype, float* master, float* m,
                         float* v, uint16_t* w_bf16, int64_t psi_pad, int32_t N,
                         const zero_adam_hparams* hp, float loss_scale, void* workspace,
                         size_t workspace_bytes_given, zero_step_result* result, void* stream) {
    if (master == nullptr && psi_pad > 0) return ZERO_ERR_ARG;
    return run_step(grads, grad_dtype, master, m, v, w_bf16, master, m, v, w_bf16, psi_pad, N, hp,
                    loss_scale, workspace, workspace_bytes_given, result, stream);
}

extern "C" int zero_step_into(const void* const* grads, int32_t grad_dtype,
                              const float* src_master, const float* src_m, const float* src_v,
                              const uint16_t* src_w_bf16, float* dst_master, float* dst_m,
                              float* dst_v, uint16_t* dst_w_bf16, int64_t psi_pad, int32_t N,
                              const zero_adam_hparams* hp, float loss_scale, void* workspace,
                              size_t workspace_bytes_given, zero_step_result* result,
                              void* stream) {
    if (psi_pad > 0 && (src_master == nullptr || dst_master == nullptr)) return ZERO_ERR_ARG;
    if (psi_pad > 0 && static_cast<const void*>(src_master) == static_cast<const void*>(dst_master))
        return ZERO_ERR_OVERLAP;
    return run_step(grads, grad_dtype, src_master, src_m, src_v, src_w_bf16, dst_master, dst_m,
                    dst_v, dst_w_bf16, psi_pad, N, hp, loss_scale, workspace,
                    workspace_bytes_given, result, stream);
}

extern "C" int zero_plan_init(zero_plan* plan, const void* const* grads, int32_t grad_dtype,
                              const float* src_master, const float* src_m, const float* src_v,
                              const uint16_t* src_w_bf16, float* dst_master, float* dst_m,
                              float* dst_v, uint16_t* dst_w_bf16, int64_t psi_pad, int32_t N,
                              const zero_adam_hparams* hp, float loss_scale, void* workspace,
                              size_t workspace_bytes_given) {
    if (psi_pad > 0 && (src_master == nullptr || dst_master == nullptr)) return ZERO_ERR_ARG;
    return plan_init(plan, grads, grad_dtype, src_master, src_m, src_v, src_w_bf16, dst_master,
                     dst_m, dst_v, dst_w_bf16, psi_pad, N, hp, loss_scale, workspace,
                     workspace_bytes_given, true);
}

extern "C" int zero_plan_init_ex(zero_plan* plan, const void* const* grads, int32_t grad_dtype,
                                 const float* src_master, const float* src_m, const float* src_v,
                                 const uint16_t* src_w_bf16, float* dst_master, float* dst_m,
                                 float* dst_v, uint16_t* dst_w_bf16, int64_t psi_pad, int32_t N,
                                 const zero_adam_hparams* hp, float loss_scale, void* workspace,
                                 size_t workspace_bytes_given, float* grad_accum) {
    if (psi_pad > 0 && (src_master == nullptr || dst_master == nullptr)) return ZERO_ERR_ARG;
    return plan_init(plan, grads, grad_dtype, src_master, src_m, src_v, src_w_bf16, dst_master,
                     dst_m, dst_v, dst_w_bf16, psi_pad, N, hp, loss_scale, workspace,
                     workspace_bytes_given, true, grad_accum);
}

namespace {

// The device address of a device-addressable buffer (device memory, or pinned
// host memory mapped for the device), or nullptr.
void* device_address(const void* p) {
    cudaPointerAttributes attr;
    if (cudaPointerGetAttributes(&attr, p) != cudaSuccess || attr.devicePointer == nullptr) {
        cudaGetLastError();  // clear the error that query may leave behind
        return nullptr;
    }
    return attr.devicePointer;
}

int set_device_policy(zero_plan* plan, zero_device_policy* policy, const float* table,
                      int64_t t_first, int32_t t_count) {
    // An in-place one-pass step cannot leave its state alone once it has run,
    // so a window miss must be caught before: only the plan's kernels check
    // it, and they all do.
    void* pol = device_address(policy);
    if (pol == nullptr) return ZERO_ERR_ARG;
    const void* tab = nullptr;
    if (table != nullptr && (tab = device_address(table)) == nullptr) return ZERO_ERR_ARG;
    plan->policy = pol;
    plan->policy_table = static_cast<const float*>(tab);
    plan->policy_t_first = t_first;
    plan->policy_t_count = t_count;
    return ZERO_OK;
}

}  // namespace

extern "C" int zero_plan_set_device_policy(zero_plan* plan, zero_device_policy* policy,
                                           int64_t t_first, int32_t t_count) {
    if (plan == nullptr || plan->state != 1 || policy == nullptr || t_first < 1 || t_count < 1 ||
        t_count > ZERO_POLICY_WINDOW || !aligned(policy, 8))
        return ZERO_ERR_ARG;
    return set_device_policy(plan, policy, nullptr, t_first, t_count);
}

extern "C" int zero_policy_table_fill(const zero_adam_hparams* hp, int64_t t_first,
                                      int64_t t_count, float* table) {
    if (table == nullptr || !valid_hparams(hp) || t_first < 1 || t_count < 1 ||
        t_count > ZERO_MAX_ELEMS || t_first - 1 > ZERO_MAX_ELEMS - t_count)
        return ZERO_ERR_ARG;
    zero_adam_hparams h = *hp;
    for (int64_t i = 0; i < t_count; ++i) {
        h.step = t_first + i;
        const Scalars s = make_scalars(&h, 1, 1.0f);
        table[2 * i] = s.step_size;
        table[2 * i + 1] = s.sbc2;
    }
    return ZERO_OK;
}

extern "C" int zero_plan_set_device_policy_table(zero_plan* plan, zero_device_policy* policy,
                                                 const float* table, int64_t t_first,
                                                 int32_t t_count) {
    if (plan == nullptr || plan->state != 1 || policy == nullptr || table == nullptr ||
        t_first < 1 || t_count < 1 || t_first - 1 > ZERO_MAX_ELEMS - t_count ||
        !aligned(policy, 8) || !aligned(table, 8))
        return ZERO_ERR_ARG;
    return set_device_policy(plan, policy, table, t_first, t_count);
}

extern "C" int zero_plan_set_pingpong(zero_plan* plan, int32_t* current_set) {
    if (plan == nullptr || plan->state != 1 || current_set == nullptr || !aligned(current_set, 4))
        return ZERO_ERR_ARG;
    // Both sets are read and written, so the step must be out of place, the
    // src set complete, and every buffer of both sets disjoint from the rest.
    if (plan->in_place) return ZERO_ERR_ARG;
    if (plan->psi_pad > 0) {
        if (plan->src_w_bf16 == nullptr) return ZERO_ERR_ARG;
        const uintptr_t n = static_cast<uintptr_t>(plan->psi_pad);
        Span sp[ZERO_MAX_RANKS + 12];
        int k = written_spans(plan, sp);
        auto add = [&](const void* ptr, uintptr_t bytes, bool written) {
            if (ptr != nullptr)
                sp[k++] = Span{reinterpret_cast<uintptr_t>(ptr),
                               reinterpret_cast<uintptr_t>(ptr) + bytes, written};
        };
        add(plan->src_master, 4 * n, true);
        add(plan->src_m, 4 * n, true);
        add(plan->src_v, 4 * n, true);
        add(plan->src_w_bf16, 2 * n, true);
        for (int i = 0; i < plan->N; ++i) add(plan->grads[i], n * grad_elem_bytes(plan->grad_dtype), false);
        if (!disjoint(sp, k)) return ZERO_ERR_OVERLAP;
    }
    cudaPointerAttributes attr;
    if (cudaPointerGetAttributes(&attr, current_set) != cudaSuccess ||
        attr.devicePointer == nullptr) {
        cudaGetLastError();
        return ZERO_ERR_ARG;
    }
    plan->current_set = attr.devicePointer;
    return ZERO_OK;
}

extern "C" int zero_plan_begin(zero_plan* plan, void* stream) { return plan_begin(plan, stream); }

extern "C" int zero_plan_bucket(zero_plan* plan, int64_t begin, int64_t end,
                                const void* const* bucket_grads, void* stream) {
    return plan_bucket(plan, begin, end, bucket_grads, stream);
}

extern "C" int zero_plan_end(zero_plan* plan, zero_step_result* result, void* stream) {
    return plan_end(plan, result, stream);
}

namespace zero_internal {
std::atomic<uint64_t> g_launches{0};
}  // namespace zero_internal

extern "C" uint64_t zero_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

extern "C" int64_t zero_debug_bounds_violations(void) {
#ifdef ZERO_DEBUG
    if (cudaDeviceSynchronize() != cudaSuccess) return -1;
    unsigned long long n = 0;
    const unsigned long long zero = 0;
    if (cudaMemcpyFromSymbol(&n, g_step_bounds_violations, sizeof n) != cudaSuccess ||
        cudaMemcpyToSymbol(g_step_bounds_violations, &zero, sizeof zero) != cudaSuccess)
        return -1;
    const int64_t g = zero_internal::gather_bounds_violations_take();
    return g < 0 ? -1 : static_cast<int64_t>(n) + g;
#else
    return -1;
#endif
}

// ------------------------------------------------------------------ no-allocation entry point
//
// For callers that cannot allocate device memory: zero_step with its
// workspace in a fixed array defined here.  The array lives in every GPU that
// loads this library until the process exits.  Host code must not pass the
// array's name to a kernel.  On the host that name stands for a host-side
// copy, so the address a kernel may use is looked up per device below.

static __device__ __align__(256) unsigned char g_noalloc_scratch[ZERO_NOALLOC_SCRATCH_BYTES];
static_assert(ZERO_NOALLOC_SCRATCH_BYTES == kGradOffset + 4 * ZERO_NOALLOC_MAX_TWO_PASS_ELEMS,
              "header size of the no-allocation scratch");

namespace {

constexpr int kMaxDevices = 256;

// Device address of g_noalloc_scratch on the current device.  It is looked
// up on the first call per device, with that device current, and then
// cached.  Returns nullptr if the lookup fails.
void* noalloc_scratch(int device) {
    static std::mutex mu;
    static void* addr[kMaxDevices] = {};
    if (device < 0 || device >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(mu);
    if (addr[device] == nullptr) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) {
            cudaGetLastError();  // leave no error behind for the caller's next call
            return nullptr;
        }
        addr[device] = p;
    }
    return addr[device];
}

}  // namespace

extern "C" int zero_step_noalloc(const void* const* grads, int32_t grad_dtype, float* master,
                                 float* m, float* v, uint16_t* w_bf16, int64_t psi_pad, int32_t N,
                                 const zero_adam_hparams* hp, float loss_scale,
                                 zero_step_result* result, void* stream) {
    // zero_step's own argument and alignment checks come first, on the host.
    // Run without a workspace, a call whose arguments pass them all stops at
    // the workspace check; only then is the size held against the array.
    if (master == nullptr && psi_pad > 0) return ZERO_ERR_ARG;
    if (hp == nullptr || micro_batches_of(hp) > 1) return ZERO_ERR_ARG;
    {
        zero_plan probe;
        const int rc = plan_init(&probe, grads, grad_dtype, master, m, v, w_bf16, master, m, v,
                                 w_bf16, psi_pad, N, hp, loss_scale, nullptr, 0, false);
        if (rc != ZERO_ERR_WORKSPACE) return rc;
    }
    if (workspace_bytes(psi_pad, hp, true) > ZERO_NOALLOC_SCRATCH_BYTES) return ZERO_ERR_TOO_LARGE;
    int device = 0;
    if (cudaGetDevice(&device) != cudaSuccess) return ZERO_ERR_CUDA;
    void* scratch = noalloc_scratch(device);
    if (scratch == nullptr) return ZERO_ERR_CUDA;
    return zero_step(grads, grad_dtype, master, m, v, w_bf16, psi_pad, N, hp, loss_scale, scratch,
                     ZERO_NOALLOC_SCRATCH_BYTES, result, stream);
}
