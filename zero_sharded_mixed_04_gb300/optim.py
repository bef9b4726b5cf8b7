"""Host-side bookkeeping around the C-ABI step.

The C ABI leaves the step counter and the loss scale to the caller.  This
module keeps them:
  - the Adam step t advances only on applied steps;
  - a dynamic loss scale halves after an overflowing (skipped) step and
    doubles after ``growth_interval`` clean steps in a row.
It also owns the device buffers of one simulated data-parallel group, all
allocated with torch:
  - N gradient buffers;
  - the FP32 master/m/v and the BF16 working weights;
  - a second set of those when the step runs out of place;
  - the workspace, and a pinned result word the device writes.
Every step runs in libzero_gb300.so; nothing here touches the data.
"""
from __future__ import annotations

import collections
import ctypes
from dataclasses import dataclass

import torch

from . import zero as Z


@dataclass
class LossScaler:
    """Dynamic loss scale: scale *= backoff after a step with a non-finite
    gradient (the clean-step count restarts), scale *= growth after
    ``interval`` clean steps in a row.  A static scale never changes."""
    scale: float = 1.0
    dynamic: bool = False
    interval: int = 2000
    backoff: float = 0.5
    growth: float = 2.0
    good_steps: int = 0

    def update(self, found_nonfinite: bool) -> None:
        if not self.dynamic:
            return
        if found_nonfinite:
            self.scale *= self.backoff
            self.good_steps = 0
            return
        self.good_steps += 1
        if self.good_steps == self.interval:
            self.scale *= self.growth
            self.good_steps = 0


class ZeroAdam:
    """The N simulated ranks' update state on one GPU, stepped through the C ABI.

    ``out_of_place`` keeps two sets of master/m/v/w and calls
    ``zero_step_into`` (the post-step state lands in the other set, which
    then becomes current).  Otherwise ``zero_step`` updates one set in place.

    ``pingpong`` (out of place only) lets the device keep which set is current
    (``zero_plan_set_pingpong``): a skipped step then leaves the current set
    current instead of copying it into the other one.  The host learns the
    current set when it next synchronises (``state()`` does).

    ``device_policy`` keeps t and the loss scale on the device, so steps need
    no host read in between.  With ``policy_table_steps`` = T as well, the bias
    corrections of t = 1 .. T come from a device table, no launch depends on
    t, and ``capture_step`` records one step as a CUDA graph to replay.
    """

    def __init__(self, psi_pad: int, N: int, grad_dtype: str = "bf16", *, lr=1e-3, beta1=0.9,
                 beta2=0.999, eps=1e-8, weight_decay=0.0, max_grad_norm=0.0,
                 skip_on_overflow=False, bucket_elems=0, loss_scale=1.0,
                 dynamic_loss_scale=False, growth_interval=2000, out_of_place=False,
                 device="cuda", master: torch.Tensor | None = None, micro_batches: int = 0,
                 host_grad_accum: bool = False, device_policy: bool = False,
                 smem_staging: int = 0, pingpong: bool = False, policy_table_steps: int = 0):
        if pingpong and not out_of_place:
            raise ValueError("ping-pong state sets need the out-of-place step")
        self.psi_pad, self.N = psi_pad, N
        self.grad_dtype = Z.ZERO_GRAD_BF16 if grad_dtype == "bf16" else Z.ZERO_GRAD_FP32
        self.hp = Z.make_hparams(lr, beta1, beta2, eps, weight_decay, max_grad_norm, 1,
                                 skip_on_overflow, bucket_elems, micro_batches)
        self.t = 0  # applied steps so far
        self.scaler = LossScaler(loss_scale, dynamic_loss_scale, growth_interval)
        self.out_of_place = out_of_place
        # smem_staging: zero_plan.smem_staging for the plan-path steps
        # (ZERO_STAGING_TMA stages every tile in shared memory by TMA bulk copies)
        self.smem_staging = smem_staging
        self.device = torch.device(device)
        sets = 2 if out_of_place else 1
        self._bufs = []
        for k in range(sets):
            p = (master.clone() if master is not None else
                 torch.zeros(psi_pad, dtype=torch.float32, device=self.device))
            self._bufs.append({
                "master": p,
                "m": torch.zeros(psi_pad, dtype=torch.float32, device=self.device),
                "v": torch.zeros(psi_pad, dtype=torch.float32, device=self.device),
                "w": torch.zeros(psi_pad, dtype=torch.int16, device=self.device),
            })
        self.cur = 0
        # host_grad_accum: the owner's FP32 gradient shard (or accumulator) lives
        # in pinned host memory and the kernels reach it over the host link;
        # steps then go through the plan entry points
        self._grad_accum_buf = None
        self.grad_accum = None
        if host_grad_accum:
            from .hostmem import HostBuffer, gpu_numa_node
            self._grad_accum_buf = HostBuffer(psi_pad, torch.float32,
                                              numa_node=gpu_numa_node(self.device))
            self.grad_accum = self._grad_accum_buf.tensor
            self.grad_accum.zero_()
        self.ws_bytes = (Z.ZERO_WORKSPACE_CONTROL_BYTES if host_grad_accum else
                         Z.zero_workspace_bytes(psi_pad, self.hp, not out_of_place))
        self.workspace = torch.empty(self.ws_bytes, dtype=torch.uint8, device=self.device)
        # device_policy: t and the loss scale live in a zero_device_policy in
        # pinned host memory that the device updates at the end of each step,
        # so steps need no host read in between
        self.policy_mem = None
        if device_policy:
            nbytes = ctypes.sizeof(Z.zero_device_policy)
            self.policy_mem = torch.zeros(nbytes, dtype=torch.uint8, pin_memory=True)
            self.policy = Z.zero_device_policy.from_address(self.policy_mem.data_ptr())
            self.policy.t = 0
            self.policy.loss_scale = loss_scale
            self.policy.good_steps = 0
            self.policy.growth_interval = growth_interval if dynamic_loss_scale else 0
            self.policy.backoff = self.scaler.backoff
            self.policy.growth = self.scaler.growth
            self._inflight = collections.deque()
        # policy_table_steps: the bias corrections of t = 1 .. policy_table_steps
        # sit in a device table (zero_plan_set_device_policy_table) instead of
        # travelling with each launch, so no launch depends on t and a captured
        # step can be replayed (capture_step); lr and the betas are fixed then
        self.policy_table = None
        if policy_table_steps > 0:
            if not device_policy:
                raise ValueError("a policy table needs the device policy")
            host = torch.empty(2 * policy_table_steps, dtype=torch.float32)
            Z.check(Z.zero_policy_table_fill(self.hp, 1, policy_table_steps, host),
                    "zero_policy_table_fill")
            self.policy_table = host.to(self.device)
        self.result_t = torch.zeros(4, dtype=torch.int32, pin_memory=True)
        self.last = None
        # pingpong: the device-kept index of the current set, in pinned memory
        self.pingpong = pingpong
        self.set_mem = torch.zeros(1, dtype=torch.int32, pin_memory=True) if pingpong else None

    # ---------------------------------------------------------------- state
    def state(self) -> dict:
        """The current master/m/v (FP32) and working weights (BF16 bits as int16).
        With ping-pong sets this waits for the device, which alone knows which
        set is current while steps are in flight."""
        if self.pingpong:
            torch.cuda.synchronize(self.device)
            self.cur = int(self.set_mem[0]) & 1
        return self._bufs[self.cur]

    def load_state(self, master, m, v, w) -> None:
        if self.pingpong:
            torch.cuda.synchronize(self.device)
            self.set_mem[0] = 0
            self.cur = 0
        s = self.state()
        s["master"].copy_(master)
        s["m"].copy_(m)
        s["v"].copy_(v)
        s["w"].copy_(w)

    # ---------------------------------------------------------------- step
    def enqueue(self, grads, stream=None, api: str = "step", bucket_events=None,
                span_events=None) -> int:
        """Enqueue one step on ``stream`` (torch's current stream by default)
        without waiting for it.  Returns the C status (ZERO_OK on success).

        api="step" calls zero_step / zero_step_into.  api="plan" enqueues the
        same kernels bucket by bucket through the plan entry points:
          - ``span_events``, a (start, end) pair of torch CUDA events, is
            recorded before the first and after the last bucket launch.
            Consecutive launches still overlap, as in zero_step.
          - ``bucket_events``, one (start, end) pair per bucket, is recorded
            around each bucket's launch instead.  The events between launches
            keep them from overlapping."""
        self.hp.step = self.t + 1
        src = self._bufs[self.cur]
        if (api == "plan" or self.grad_accum is not None or self.policy_mem is not None
                or self.smem_staging or self.pingpong):
            return self._enqueue_plan(grads, src, stream, bucket_events, span_events)
        if self.out_of_place:
            dst = self._bufs[1 - self.cur]
            rc = Z.zero_step_into(grads, self.grad_dtype, src["master"], src["m"], src["v"],
                                  src["w"], dst["master"], dst["m"], dst["v"], dst["w"],
                                  self.psi_pad, self.N, self.hp, self.scaler.scale,
                                  self.workspace, self.ws_bytes, self.result_t, stream)
        else:
            rc = Z.zero_step(grads, self.grad_dtype, src["master"], src["m"], src["v"], src["w"],
                             self.psi_pad, self.N, self.hp, self.scaler.scale, self.workspace,
                             self.ws_bytes, self.result_t, stream)
        Z.check(rc, "zero_step")
        if self.out_of_place:
            self.cur = 1 - self.cur  # dst always holds the post-step state
        return rc

    def bucket_bounds(self) -> list[tuple[int, int]]:
        b = self.hp.bucket_elems or self.psi_pad
        return [(b0, min(self.psi_pad, b0 + b)) for b0 in range(0, self.psi_pad, b)]

    def _sets(self):
        """(src, dst) buffer sets of the next step's plan: with ping-pong sets
        always set 0 and set 1 (the device picks which one it reads)."""
        if self.pingpong:
            return self._bufs[0], self._bufs[1]
        src = self._bufs[self.cur]
        return src, (self._bufs[1 - self.cur] if self.out_of_place else src)

    def _after_enqueue(self) -> None:
        # with ping-pong sets the device flips the current set itself
        if self.out_of_place and not self.pingpong:
            self.cur = 1 - self.cur

    def _enqueue_plan(self, grads, src, stream, bucket_events, span_events=None) -> int:
        src, dst = self._sets()
        plan = Z.zero_plan()
        Z.check(Z.zero_plan_init_ex(plan, grads, self.grad_dtype, src["master"], src["m"],
                                    src["v"], src["w"], dst["master"], dst["m"], dst["v"], dst["w"],
                                    self.psi_pad, self.N, self.hp, self.scaler.scale,
                                    self.workspace, self.ws_bytes, self.grad_accum),
                "zero_plan_init")
        # nothing but bucket launches goes between the buckets unless events
        # are recorded around each one
        plan.overlap_buckets = 0 if bucket_events is not None else 1
        plan.smem_staging = self.smem_staging
        self._apply_policy(plan, stream)
        Z.check(Z.zero_plan_begin(plan, stream), "zero_plan_begin")
        s = stream if stream is not None else torch.cuda.current_stream(self.device)
        if span_events is not None:
            span_events[0].record(s)
        n0 = Z.zero_launch_count()
        for k, (b0, b1) in enumerate(self.bucket_bounds()):
            if bucket_events is not None:
                bucket_events[k][0].record(s)
            Z.check(Z.zero_plan_bucket(plan, b0, b1, None, stream), "zero_plan_bucket")
            if bucket_events is not None:
                bucket_events[k][1].record(s)
        if span_events is not None:
            span_events[1].record(s)
        # kernel launches of the first pass (the library splits long ranges)
        self.first_pass_launches = Z.zero_launch_count() - n0
        rc = Z.check(Z.zero_plan_end(plan, self.result_t, stream), "zero_plan_end")
        self._note_enqueued(s)
        self._after_enqueue()
        return rc

    # ---------------------------------------------------------------- accumulation
    def enqueue_accumulated(self, micro_grads, stream=None, span_events=None) -> int:
        """Enqueue one step whose gradient is accumulated over the micro-batches
        in ``micro_grads`` (a list of k lists of N gradient buffers; k must equal
        the micro_batches this object was made with).  Each micro-batch's buckets
        are reduce-scattered into the owner's FP32 accumulator in turn; the
        update follows the last one (in the same pass when the step needs no
        second pass).  ``span_events``: two events recorded around all the
        micro-batches' launches, or three, the middle one recorded before the
        last micro-batch's.  ``pass_launches`` then holds the kernel launches of
        each micro-batch's pass."""
        k = max(1, self.hp.micro_batches)
        if len(micro_grads) != k:
            raise ValueError(f"expected {k} micro-batches, got {len(micro_grads)}")
        self.hp.step = self.t + 1
        src, dst = self._sets()
        plan = Z.zero_plan()
        Z.check(Z.zero_plan_init_ex(plan, micro_grads[0], self.grad_dtype, src["master"],
                                    src["m"], src["v"], src["w"], dst["master"], dst["m"],
                                    dst["v"], dst["w"], self.psi_pad, self.N, self.hp,
                                    self.scaler.scale, self.workspace, self.ws_bytes,
                                    self.grad_accum), "zero_plan_init")
        plan.overlap_buckets = 1
        self._apply_policy(plan, stream)
        Z.check(Z.zero_plan_begin(plan, stream), "zero_plan_begin")
        s = stream if stream is not None else torch.cuda.current_stream(self.device)
        if span_events is not None:
            span_events[0].record(s)
        n0 = Z.zero_launch_count()
        self.pass_launches = []
        for i, grads in enumerate(micro_grads):
            if span_events is not None and len(span_events) == 3 and i == k - 1:
                span_events[1].record(s)
            n1 = Z.zero_launch_count()
            for b0, b1 in self.bucket_bounds():
                Z.check(Z.zero_plan_bucket(plan, b0, b1, [g[b0:b1] for g in grads], stream),
                        "zero_plan_bucket")
            self.pass_launches.append(Z.zero_launch_count() - n1)
        if span_events is not None:
            span_events[-1].record(s)
        self.first_pass_launches = Z.zero_launch_count() - n0
        rc = Z.check(Z.zero_plan_end(plan, self.result_t, stream), "zero_plan_end")
        self._note_enqueued(s)
        self._after_enqueue()
        return rc

    def step_accumulated(self, micro_grads, stream=None) -> dict:
        self.enqueue_accumulated(micro_grads, stream)
        return self.finish(stream)

    def step_accumulated_async(self, micro_grads, stream=None, span_events=None) -> dict | None:
        """step_accumulated without the wait, under the same rule as step_async."""
        self.enqueue_accumulated(micro_grads, stream, span_events)
        if self.needs_result:
            return self.finish(stream)
        if self.policy_mem is None:
            self.t += 1
        return None

    # ---------------------------------------------------------------- host gradients
    def make_slots(self, bucket_elems: int | None = None) -> list[list[torch.Tensor]]:
        """Two device staging slots, each holding one bucket of all N ranks'
        gradients: the two-buffer pattern (one slot read while the other refills)."""
        b = bucket_elems or self.hp.bucket_elems or self.psi_pad
        dt = torch.bfloat16 if self.grad_dtype == Z.ZERO_GRAD_BF16 else torch.float32
        return [[torch.empty(b, dtype=dt, device=self.device) for _ in range(self.N)]
                for _ in range(2)]

    def enqueue_from_host(self, host_grads, slots, copy_stream, stream=None) -> int:
        """Enqueue one step whose N gradients sit in pinned host memory.  Bucket
        k is copied into slot k % 2 on ``copy_stream`` while the compute stream
        reduces bucket k - 1 from the other slot.  A slot is refilled only once
        the bucket that used it has been read."""
        self.hp.step = self.t + 1
        src, dst = self._sets()
        s = stream if stream is not None else torch.cuda.current_stream(self.device)
        plan = Z.zero_plan()
        Z.check(Z.zero_plan_init_ex(plan, [None] * self.N, self.grad_dtype, src["master"],
                                    src["m"], src["v"], src["w"], dst["master"], dst["m"],
                                    dst["v"], dst["w"], self.psi_pad, self.N, self.hp,
                                    self.scaler.scale, self.workspace, self.ws_bytes,
                                    self.grad_accum), "zero_plan_init")
        plan.smem_staging = self.smem_staging
        self._apply_policy(plan, s)
        Z.check(Z.zero_plan_begin(plan, s), "zero_plan_begin")
        if not hasattr(self, "_slot_events"):
            # freed[k] is recorded after the last read of slot k, also across steps
            self._slot_events = ([torch.cuda.Event(), torch.cuda.Event()],
                                 [torch.cuda.Event(), torch.cuda.Event()])
        loaded, freed = self._slot_events
        b = slots[0][0].numel()
        for k, b0 in enumerate(range(0, self.psi_pad, b)):
            b1 = min(self.psi_pad, b0 + b)
            slot = slots[k % 2]
            copy_stream.wait_event(freed[k % 2])  # no-op before the first record
            with torch.cuda.stream(copy_stream):
                for i in range(self.N):
                    slot[i][:b1 - b0].copy_(host_grads[i][b0:b1], non_blocking=True)
            loaded[k % 2].record(copy_stream)
            s.wait_event(loaded[k % 2])
            Z.check(Z.zero_plan_bucket(plan, b0, b1, slot, s), "zero_plan_bucket")
            freed[k % 2].record(s)
        rc = Z.check(Z.zero_plan_end(plan, self.result_t, s), "zero_plan_end")
        self._note_enqueued(s)
        self._after_enqueue()
        return rc

    def _apply_policy(self, plan, stream) -> None:
        if self.pingpong:
            Z.check(Z.zero_plan_set_pingpong(plan, self.set_mem), "zero_plan_set_pingpong")
        if self.policy_table is not None:
            Z.check(Z.zero_plan_set_device_policy_table(plan, self.policy_mem, self.policy_table,
                                                        1, self.policy_table.numel() // 2),
                    "zero_plan_set_device_policy_table")
        elif self.policy_mem is not None:
            t_first, t_count = self._policy_window(stream)
            Z.check(Z.zero_plan_set_device_policy(plan, self.policy_mem, t_first, t_count),
                    "zero_plan_set_device_policy")

    def _note_enqueued(self, s) -> None:
        # only a window of bias corrections depends on how many steps are in flight
        if self.policy_mem is not None and self.policy_table is None:
            ev = torch.cuda.Event()
            ev.record(s)
            self._inflight.append(ev)

    def _policy_window(self, stream=None) -> tuple[int, int]:
        """The t values the next step may see on the device: from the policy's
        t, read after the completed steps are known, up to one more per step
        still in flight."""
        while self._inflight and self._inflight[0].query():
            self._inflight.popleft()
        while len(self._inflight) >= Z.ZERO_POLICY_WINDOW - 1:
            self._inflight.popleft().synchronize()
        t_read = int(self.policy.t)
        return t_read + 1, len(self._inflight) + 1

    def finish(self, stream=None) -> dict:
        """Wait for the last enqueued step, read its result and advance the
        host bookkeeping (t and the loss scale)."""
        s = stream if stream is not None else torch.cuda.current_stream(self.device)
        s.synchronize()
        raw = self.result_t.clone()
        status = int(raw[0])
        found = bool(int(raw[1]))
        norm = float(raw[2:3].view(torch.float32)[0])
        coef = float(raw[3:4].view(torch.float32)[0])
        Z.check(status, "zero_step (device)")
        applied = status == Z.ZERO_OK
        if self.policy_mem is not None:
            self._inflight.clear()               # the stream is idle
            self.t = int(self.policy.t)
            self.scaler.scale = float(self.policy.loss_scale)
            self.scaler.good_steps = int(self.policy.good_steps)
        else:
            if applied:
                self.t += 1
            self.scaler.update(found)
        self.last = {"applied": applied, "found_nonfinite": found, "grad_norm": norm,
                     "clip_coef": coef, "status": status}
        return self.last

    @property
    def needs_result(self) -> bool:
        """Whether the host must read each step's outcome before the next one.
        It must when a step can be skipped (t then does not advance) or the
        loss scale reacts to overflow.  Otherwise every step applies and the
        host can run ahead of the device."""
        if self.policy_mem is not None:
            return False  # the device keeps t and the loss scale
        return bool(self.hp.skip_on_overflow) or self.scaler.dynamic

    def step_async(self, grads, stream=None, api: str = "step", span_events=None) -> dict | None:
        """Like step(), but without waiting when the outcome cannot change the
        host's bookkeeping (see needs_result): t advances at once and None is
        returned.  last_result() reads the latest outcome."""
        self.enqueue(grads, stream, api, None, span_events)
        if self.needs_result:
            return self.finish(stream)
        if self.policy_mem is None:
            self.t += 1
        return None

    def last_result(self, stream=None) -> dict:
        """Wait for the stream and read the most recent step's outcome, without
        changing t or the loss scale."""
        s = stream if stream is not None else torch.cuda.current_stream(self.device)
        s.synchronize()
        raw = self.result_t.clone()
        Z.check(int(raw[0]), "zero_step (device)")
        return {"applied": int(raw[0]) == Z.ZERO_OK, "found_nonfinite": bool(int(raw[1])),
                "grad_norm": float(raw[2:3].view(torch.float32)[0]),
                "clip_coef": float(raw[3:4].view(torch.float32)[0]), "status": int(raw[0])}

    def step(self, grads, stream=None, api: str = "step", bucket_events=None,
             span_events=None) -> dict:
        self.enqueue(grads, stream, api, bucket_events, span_events)
        return self.finish(stream)


    # ---------------------------------------------------------------- CUDA graphs
    def capture_step(self, grads, stream=None) -> torch.cuda.CUDAGraph:
        """One step on ``grads`` (N device buffers) captured as a CUDA graph.
        Each replay runs one more step with whatever the buffers then hold:
        refill them on the replaying stream, then replay.  The step keeps all
        of its host state on the device (t, the loss scale, the bias
        corrections from the policy table and, out of place, the current
        ping-pong set), so replays need no host work in between; the host
        catches up at finish_pending() or state().  Needs the device policy
        with a policy table, and ping-pong sets when out of place."""
        if self.policy_table is None:
            raise ValueError("capture_step needs device_policy and policy_table_steps")
        if self.out_of_place and not self.pingpong:
            raise ValueError("capture_step needs ping-pong sets when out of place")
        if self.hp.micro_batches > 1:
            raise ValueError("capture_step takes one batch")
        s = stream if stream is not None else torch.cuda.Stream(self.device)
        s.wait_stream(torch.cuda.current_stream(self.device))
        graph = torch.cuda.CUDAGraph()
        # relaxed: the plan queries pointer attributes while it is captured
        with torch.cuda.graph(graph, stream=s, capture_error_mode="relaxed"):
            self._enqueue_plan(grads, None, s, None)
        return graph

    # ---------------------------------------------------------------- checkpoint
    def finish_pending(self) -> None:
        """Wait for every enqueued step and bring t and the loss scale up to
        date (with a device policy they live on the device)."""
        torch.cuda.synchronize(self.device)
        if self.policy_mem is not None:
            self._inflight.clear()
            self.t = int(self.policy.t)
            self.scaler.scale = float(self.policy.loss_scale)
            self.scaler.good_steps = int(self.policy.good_steps)

    def state_dict(self) -> dict:
        """Everything a later step depends on, on the host: the current
        master/m/v and working weights, the step counter and the loss-scale
        state."""
        self.finish_pending()
        st = self.state()
        return {"master": st["master"].cpu(), "m": st["m"].cpu(), "v": st["v"].cpu(),
                "w": st["w"].cpu(), "t": self.t, "loss_scale": self.scaler.scale,
                "good_steps": self.scaler.good_steps, "psi_pad": self.psi_pad, "N": self.N}

    def load_state_dict(self, sd: dict) -> None:
        if sd["psi_pad"] != self.psi_pad or sd["N"] != self.N:
            raise ValueError("checkpoint of a different layout")
        self.finish_pending()
        self.load_state(sd["master"], sd["m"], sd["v"], sd["w"])
        self.t = int(sd["t"])
        self.scaler.scale = float(sd["loss_scale"])
        self.scaler.good_steps = int(sd["good_steps"])
        if self.policy_mem is not None:
            self.policy.t = self.t
            self.policy.loss_scale = self.scaler.scale
            self.policy.good_steps = self.scaler.good_steps


class Zero3Views:
    """ZeRO-3 per-layer gather with two views: before layer i runs, layer i + 1
    is gathered into the other view on a side stream; a view is reused only
    after the layer that held it ran (released).  The layers are flat ranges
    [begin, end) of the vector whose BF16 shards are ``shards`` (N device
    buffers of ``shard`` elements, e.g. the owners' slices of a step's
    working weights).

    ``side_streams``: 1 gathers every layer on one side stream, each gather
    chained to the one before it; 2 gives each view its own side stream, so
    the gathers of neighbouring layers (which fill different views) may run at
    the same time, while a view is still refilled only after its previous
    layer ran.  Either way at most two layers are gathered at once, so the
    peak ledger (zero3_peak_bytes) holds."""

    def __init__(self, shards, shard: int, layers, device="cuda", side_streams: int = 2):
        if side_streams not in (1, 2):
            raise ValueError("side_streams is 1 or 2")
        self.shards = list(shards)
        self.N = len(self.shards)
        self.shard = shard
        self.layers = [(int(b), int(e)) for b, e in layers]
        self.device = torch.device(device)
        most = max((e - b for b, e in self.layers), default=0)
        self.views = [torch.empty(max(most, 1), dtype=torch.int16, device=self.device)
                      for _ in range(2)]
        first = torch.cuda.Stream(self.device)
        self.sides = [first, torch.cuda.Stream(self.device) if side_streams == 2 else first]
        self.side = first
        self.gathered = [torch.cuda.Event(), torch.cuda.Event()]
        self.released = [torch.cuda.Event(), torch.cuda.Event()]

    def _gather(self, i: int) -> None:
        b, e = self.layers[i]
        slot = i % 2
        side = self.sides[slot]
        if i >= 2:
            # layers 0 and 1 refill views that the previous pass released
            # before this pass began; the side streams' wait for the caller's
            # stream at the start of the pass already orders them
            side.wait_event(self.released[slot])
        # One side stream: after the first layer of a pass the kernel before
        # this gather is the previous layer's gather, which reads the shards
        # and writes the other view, so this one may start while it drains.
        # Two: the kernel before it on its stream is the gather of layer i - 2,
        # into this same view, but the wait just above (for the use of that
        # layer) is a complete dependency and orders it first.
        one_stream = self.sides[0] is self.sides[1]
        flags = Z.ZERO3_GATHER_OVERLAP_PREVIOUS if i >= (1 if one_stream else 2) else 0
        Z.check(Z.zero3_gather(self.shards, self.N, self.shard, b, e, self.views[slot],
                               side, flags=flags), "zero3_gather")
        self.gathered[slot].record(side)

    def run(self, use, stream=None) -> None:
        """Calls use(i, view) for every layer in order, on ``stream``, where view
        is the layer's gathered BF16 values (int16 bits)."""
        s = stream if stream is not None else torch.cuda.current_stream(self.device)
        if not self.layers:
            return
        for side in {id(x): x for x in self.sides}.values():
            side.wait_stream(s)  # the shards are ready on s
        self._gather(0)
        for i, (b, e) in enumerate(self.layers):
            if i + 1 < len(self.layers):
                self._gather(i + 1)           # prefetch into the other view
            slot = i % 2
            s.wait_event(self.gathered[slot])
            use(i, self.views[slot][:e - b])
            self.released[slot].record(s)     # the view may be refilled

    def capture(self, use=None):
        """One pass of run() recorded as a CUDA graph, for a layer list that is
        the same every pass.  graph.replay() then issues every gather, wait and
        use(i, view) of the pass with no host work per layer.  The graph holds
        the shards', views' and layers' addresses, so it reads whatever the
        shards hold when it is replayed.  use must be capturable: device work
        only, no host synchronisation.  One eager pass runs first."""
        fn = use if use is not None else (lambda i, view: None)
        cur = torch.cuda.current_stream(self.device)
        cap = torch.cuda.Stream(self.device)
        cap.wait_stream(cur)
        with torch.cuda.stream(cap):
            self.run(fn, cap)           # warm-up: caches the launch shapes
        cap.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=cap):
            self.run(fn, cap)
        cur.wait_stream(cap)
        return graph
