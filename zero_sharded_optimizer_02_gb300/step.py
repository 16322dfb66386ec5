"""Host side of the ZeRO-DP optimizer step: buffers, launch, skip and commit.

``DataParallelStep`` holds the fp32 optimizer state of one or more ranks of a
data-parallel group ("ZeRO: Memory Optimizations Toward Training Trillion
Parameter Models", section "ZeRO-DP": each rank holds and updates only its
1/Nd of the state) in device memory, launches the library's step for each of
them and applies the global decision: if any rank's reduced gradient holds an
inf or NaN, every rank keeps its previous state, gathered parameters and step
count; otherwise every rank commits.  The state is double-buffered (``cur`` is
read, ``next`` is written), so a skip costs no extra pass over the gradients
and committing is a buffer swap.

torch is used for device memory, streams and (optionally) the one-word OR of
the skip flag over a process group; all optimizer arithmetic runs in the CUDA
kernels behind the C ABI.
"""
from __future__ import annotations

import torch

from . import _abi

_TORCH_DTYPES = {"f16": torch.float16, "bf16": torch.bfloat16}


def _collective_device(group, device):
    import torch.distributed as dist
    if dist.get_backend(group) == "nccl":
        return device if device is not None else torch.device("cuda", torch.cuda.current_device())
    return torch.device("cpu")


def global_skip(local_bad: bool, group=None, device=None) -> bool:
    """The global skip decision: True if any rank of ``group`` saw a nonfinite
    reduced gradient (a one-word MAX all-reduce; identity without a group)."""
    if group is None:
        return bool(local_bad)
    import torch.distributed as dist
    word = torch.tensor([int(bool(local_bad))], dtype=torch.int32,
                        device=_collective_device(group, device))
    dist.all_reduce(word, op=dist.ReduceOp.MAX, group=group)
    return int(word.item()) != 0


def max_over_ranks(x: float, group=None, device=None) -> float:
    """The maximum of a per-rank float over ``group`` (identity without one)."""
    if group is None:
        return float(x)
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=_collective_device(group, device))
    dist.all_reduce(t, op=dist.ReduceOp.MAX, group=group)
    return float(t.item())


def sum_over_ranks(x: int, group=None, device=None) -> int:
    """The sum of a per-rank count over ``group`` (identity without one)."""
    if group is None:
        return int(x)
    import torch.distributed as dist
    t = torch.tensor([int(x)], dtype=torch.int64, device=_collective_device(group, device))
    dist.all_reduce(t, op=dist.ReduceOp.SUM, group=group)
    return int(t.item())


def data_parallel_rank(first_rank: int, process_rank: int, nd: int) -> int:
    """The data-parallel rank a process runs: process k of a launch runs rank
    first_rank + k of the emulated Nd-way group."""
    r = first_rank + process_rank
    if not 0 <= r < nd:
        raise ValueError(f"process {process_rank} maps to rank {r}, outside 0..{nd - 1}")
    return r


class RankState:
    """Double- (or, pipelined, triple-) buffered fp32 state (master, m, v) of
    one rank's shard."""

    def __init__(self, layout: _abi.Layout, device, nbuf: int = 2):
        self.layout = layout
        # One [3, pitch] block per buffer; pitch is a multiple of 8 elements,
        # so every row starts 32-byte aligned.
        pitch = max(int(layout.row_pitch), 8)
        self.bufs = [torch.zeros(3, pitch, dtype=torch.float32, device=device)
                     for _ in range(nbuf)]
        self.states = [_abi.state(b[0], b[1], b[2]) for b in self.bufs]
        self.cur = 0

    def tensors(self, which: str = "cur"):
        i = self.cur if which == "cur" else 1 - self.cur
        n = int(self.layout.length)
        b = self.bufs[i]
        return b[0, :n], b[1, :n], b[2, :n]

    def load(self, master, m, v) -> None:
        for row, src in zip(self.bufs[self.cur], (master, m, v)):
            row[:src.numel()].copy_(src)


class DataParallelStep:
    """The ZeRO-DP shard step for a set of ranks sharing one skip decision.

    psi, nd      flat parameter count and data-parallel degree
    ranks        the ranks held here (all of range(nd) for full emulation)
    gathered     "full": one flat fp16/bf16 buffer of nd * S parameters that
                 every rank writes its slot of; "slot": one S-element buffer
                 per rank (the persistent parameters of a ZeRO-3 rank);
                 "pitched": the ranks' slots as rows of one [nd, pitch] buffer
                 (what zero_gather_range collects a layer from)
    fused        zero_step_shard (default) or zero_step_shard_unfused
    process_group  if given, the skip flag is OR-ed over it every step
    gathered_on_host  keep the gathered buffers in page-locked host memory:
                 the kernels write the cast parameters there in place over
                 the host link, so they reach the host with no copy of
                 their own
    row_align    the row pitch of the layouts (and of the state rows) is S
                 rounded up to this many elements: 8, the default, is the
                 least the kernels accept; 512 puts every 2-byte gradient
                 row on a 1 KB boundary, which streams faster when the
                 shard's own pitch leaves rows only 32-byte aligned
    """

    def __init__(self, psi: int, nd: int, ranks, grad_dtype: str, hparams: dict,
                 loss_scale: float, bucket: int, device="cuda", gathered: str = "full",
                 fused: bool = True, process_group=None, row_align: int = 8, stream=None,
                 gathered_on_host: bool = False):
        self.psi, self.nd, self.ranks = psi, nd, list(ranks)
        self.grad_dtype = grad_dtype
        self.hp = dict(hparams)
        self.loss_scale = float(loss_scale)
        self.bucket = int(bucket)
        self.device = torch.device(device)
        self.fused = fused
        self.pg = process_group
        self.layouts = {r: _abi.zero_partition_layout(psi, nd, r, row_align) for r in self.ranks}
        self.state = {r: RankState(self.layouts[r], self.device) for r in self.ranks}
        if gathered not in ("full", "pitched", "slot"):
            raise ValueError(gathered)
        self.gathered_mode = gathered
        self.gathered_on_host = bool(gathered_on_host)
        self.gathered = [self._new_gathered() for _ in range(2)]
        self.gcur = 0
        self.stream = stream if stream is not None else torch.cuda.current_stream(self.device)
        self.flag = torch.zeros(1, dtype=torch.int32, device=self.device)
        self.flag_host = torch.zeros(1, dtype=torch.int32, pin_memory=self.device.type == "cuda")
        self.t = 0
        self.skipped_steps = []
        self.cb = None
        self.cb_elems = 0
        if not fused:
            self.cb_elems = min(self.bucket, int(self.layouts[self.ranks[0]].shard_elems)) + 4
            self.cb = torch.empty(self.cb_elems, dtype=torch.float32, device=self.device)
        self.h = _abi.adamw(self.hp["lr"], self.hp["beta1"], self.hp["beta2"], self.hp["eps"],
                            self.hp["weight_decay"], 1)

    # -- buffers -------------------------------------------------------------

    def _new_gathered(self):
        """One gathered buffer set (zeroed) in the configured layout and memory."""
        tdt = _TORCH_DTYPES[self.grad_dtype]
        s = int(self.layouts[self.ranks[0]].shard_elems)
        where = {"dtype": tdt, "device": "cpu", "pin_memory": True} if self.gathered_on_host \
            else {"dtype": tdt, "device": self.device}
        if self.gathered_mode == "full":
            return torch.zeros(self.nd * s + 8, **where)
        if self.gathered_mode == "pitched":
            pitch = int(self.layouts[self.ranks[0]].row_pitch)
            return torch.zeros(self.nd, max(pitch, 8), **where)
        return {r: torch.zeros(max(s, 1) + 8, **where) for r in self.ranks}

    def gathered_view(self, rank=None, which: str = "cur") -> torch.Tensor:
        i = self.gcur if which == "cur" else 1 - self.gcur
        if self.gathered_mode in ("full", "pitched"):
            return self.gathered[i]
        return self.gathered[i][rank]

    def _gathered_target(self, r, i):
        if self.gathered_mode == "full":
            return self.gathered[i], int(self.layouts[r].begin)
        if self.gathered_mode == "pitched":
            return self.gathered[i], r * int(self.gathered[i].shape[1])
        return self.gathered[i][r], 0

    # -- the step ------------------------------------------------------------

    def launch(self, grads: dict) -> int:
        """Launch the step of every held rank (cur -> next) on ``self.stream``.
        ``grads[r]`` is the _abi.Grads descriptor of rank r's contributions.
        Returns the number of kernel launches issued."""
        self.h.step = self.t + 1
        nxt = 1 - self.gcur
        launches = 0
        for r in self.ranks:
            st = self.state[r]
            L = self.layouts[r]
            gbuf, goff = self._gathered_target(r, nxt)
            s_in, s_out = st.states[st.cur], st.states[1 - st.cur]
            if self.fused:
                _abi.zero_step_shard(grads[r], L, s_in, s_out, gbuf, goff, self.bucket,
                                     self.loss_scale, self.h, self.flag, self.stream)
            else:
                _abi.zero_step_shard_unfused(grads[r], L, s_in, s_out, gbuf, goff, self.bucket,
                                             self.loss_scale, self.h, self.cb, self.cb_elems,
                                             self.flag, self.stream)
            n = int(L.length)
            count = _abi.fused_launch_count if self.fused else _abi.unfused_launch_count
            launches += count(n, self.bucket, int(grads[r].offset))
        return launches

    def decide(self) -> bool:
        """Read the nonfinite flag (OR-ed over the process group if any).

        If a device wait of the step expired (a host-fed step's bucket wait,
        or a step kernel's pipeline wait), every rank still takes part in the
        decision, where it counts as a skip, and then this rank raises
        ZeroError (ZERO_ERR_TIMEOUT): the step is not committed, the committed
        state is untouched, and the flag and status words are cleared so the
        next step can run."""
        with torch.cuda.stream(self.stream):
            self.flag_host.copy_(self.flag, non_blocking=True)
        self.stream.synchronize()
        word = int(self.flag_host[0])
        status = _abi.ZERO_OK
        if getattr(self, "_fed_pending", False):
            self._fed_pending = False
            status = int(self._status.item())
        expired = status != _abi.ZERO_OK or bool(word & _abi.ZERO_STEP_FLAG_WAIT_TIMEOUT)
        # every rank takes part in the decision before any rank raises
        skip = global_skip(word != 0 or expired, self.pg, self.device)
        if expired:
            with torch.cuda.stream(self.stream):
                self.flag.zero_()
                if status != _abi.ZERO_OK:
                    self._status.zero_()
            self.stream.synchronize()
            raise _abi.ZeroError(_abi.ZERO_ERR_TIMEOUT,
                                 "bucket-ready step (a bucket never arrived)"
                                 if status != _abi.ZERO_OK else "step kernel")
        return skip

    def commit(self, skipped: bool) -> None:
        self.skipped_steps.append(skipped)
        if skipped:
            with torch.cuda.stream(self.stream):
                self.flag.zero_()   # the flag is sticky; clear it only after a skip
            return
        for st in self.state.values():
            st.cur = 1 - st.cur
        self.gcur = 1 - self.gcur
        self.t += 1

    # -- gradients fed from host memory, bucket by bucket ----------------------

    def launch_host_fed(self, rank: int, host_rows, dev_grads, stream_bucket: int,
                        copy_stream, timeout_ns: int = 10_000_000_000) -> int:
        """Launch rank's step with its gradients still in (pinned) host memory:
        the bucket-ready kernel runs on ``self.stream`` while the feeder lands
        each bucket's contributions on ``copy_stream`` and marks it ready, so
        the optimizer overlaps the transfer.  ``host_rows`` is [nd, m] pinned
        (contributor j's shard at row j); ``dev_grads`` the Grads descriptor of
        the device rows they land in.  Returns the kernel launches issued.
        If a bucket's wait (timeout_ns) expires, decide() raises ZeroError
        (ZERO_ERR_TIMEOUT) for this step."""
        L = self.layouts[rank]
        n = int(L.length)
        nb = -(-n // stream_bucket) if n else 0
        if not hasattr(self, "_ready") or self._ready.numel() < max(nb, 1):
            self._ready = torch.zeros(max(nb, 1), dtype=torch.int32, device=self.device)
            self._epoch = 0
            self._epoch_host = torch.zeros(1, dtype=torch.int32, pin_memory=True)
            self._status = torch.zeros(1, dtype=torch.int32, device=self.device)
        if getattr(self, "_feed_done", None) is not None:
            # the previous feed's copies read _epoch_host; they are done unless
            # that step timed out, and must be before it is overwritten
            self._feed_done.synchronize()
        self._epoch += 1
        self._epoch_host[0] = self._epoch
        self.h.step = self.t + 1
        st = self.state[rank]
        gbuf, goff = self._gathered_target(rank, 1 - self.gcur)
        start = torch.cuda.Event()
        start.record(self.stream)
        copy_stream.wait_event(start)      # the feed starts after earlier work on self.stream
        _abi.zero_step_shard_streamed(dev_grads, L, st.states[st.cur], st.states[1 - st.cur],
                                      gbuf, goff, stream_bucket, self.loss_scale, self.h,
                                      self._ready, self._epoch, timeout_ns, self.flag,
                                      self._status, self.stream)
        _abi.zero_feed_buckets(host_rows, int(host_rows.shape[1]), dev_grads, n, stream_bucket,
                               self._ready, self._epoch_host, copy_stream)
        self._feed_done = torch.cuda.Event()
        self._feed_done.record(copy_stream)
        self._fed_pending = True
        return _abi.streamed_launch_count(n, stream_bucket, int(dev_grads.nd),
                                          int(dev_grads.offset))

    def host_fed_status(self) -> int:
        """ZERO_OK, or ZERO_ERR_TIMEOUT if a bucket never arrived (read after
        the stream work completed)."""
        return int(self._status.item()) if hasattr(self, "_status") else 0

    # -- sharded checkpoints ---------------------------------------------------

    def checkpoint_paths(self, directory: str, nd: int | None = None) -> list:
        import os
        nd = self.nd if nd is None else nd
        return [os.path.join(directory, f"zero_rank{r:05d}_of_{nd:05d}.zck") for r in range(nd)]

    def save_checkpoint(self, directory: str) -> list:
        """Each held rank writes its committed state to its own file."""
        import os
        os.makedirs(directory, exist_ok=True)
        paths = self.checkpoint_paths(directory)
        h = _abi.adamw(self.hp["lr"], self.hp["beta1"], self.hp["beta2"], self.hp["eps"],
                       self.hp["weight_decay"], self.t)
        self.stream.synchronize()
        for r in self.ranks:
            host = [t.cpu().numpy() for t in self.state[r].tensors("cur")]
            _abi.zero_checkpoint_save(paths[r], self.layouts[r], h, *host)
        return [paths[r] for r in self.ranks]

    def load_checkpoint(self, paths: list) -> None:
        """Loads every held rank's state from a checkpoint saved with
        len(paths) ranks (resharding if that differs from nd)."""
        import numpy as np
        step = None
        for r in self.ranks:
            n = int(self.layouts[r].length)
            host = [np.empty(max(n, 1), np.float32) for _ in range(3)]
            h = _abi.zero_checkpoint_load(paths, self.layouts[r], *host)
            step = int(h.step)
            with torch.cuda.stream(self.stream):
                self.state[r].load(*(torch.from_numpy(a[:n]) for a in host))
        self.stream.synchronize()
        self.t = step

    def step(self, grads: dict) -> bool:
        """One full step: launch, global decision, commit.  Returns True if skipped."""
        self.launch(grads)
        skipped = self.decide()
        self.commit(skipped)
        return skipped


class PipelinedStep(DataParallelStep):
    """DataParallelStep whose host never stalls the GPU between steps.

    Up to ``depth`` steps are launched ahead of the last decided one, each on
    its predecessor's output (speculating that every undecided step commits);
    the host waits only for the oldest undecided step's flag.  State and
    parameters need depth + 2 buffers (committed, and one per step in
    flight), and the flag alternates between depth + 1 words.  If a step
    turns out to be skipped, the committed state stays, the speculative steps
    built on it are discarded and run again from the committed state, so
    every step's result and the skip rule are exactly those of
    DataParallelStep.  The flag words are copied to the host on a side
    stream after each step's kernels, so consecutive steps' kernels run back
    to back, and depth 2 leaves the host a whole step of slack.  Gradient
    buffers must stay unchanged until the step that reads them has been
    decided.

    Use: ``launch(grads)`` for each step, then ``finish()`` once; both return
    the decided steps' skip flags in order.
    """

    def __init__(self, *args, depth: int = 2, **kwargs):
        kwargs.setdefault("gathered", "slot")
        super().__init__(*args, **kwargs)
        if depth < 1:
            raise ValueError("depth must be at least 1")
        self.depth = depth
        nbuf = depth + 2
        for r in self.ranks:
            old = self.state[r]
            self.state[r] = RankState(self.layouts[r], self.device, nbuf=nbuf)
            self.state[r].bufs[0].copy_(old.bufs[old.cur])
            self.state[r].states = [_abi.state(b[0], b[1], b[2]) for b in self.state[r].bufs]
        self.gathered = [self.gathered[self.gcur]] + [self._new_gathered()
                                                      for _ in range(nbuf - 1)]
        self.gcur = 0
        self.flags = torch.zeros(depth + 1, dtype=torch.int32, device=self.device)
        self.flags_host = torch.zeros(depth + 1, dtype=torch.int32, pin_memory=True)
        # the flag words travel to the host on a side stream, so the next
        # step's kernels never wait behind a copy
        self.flag_stream = torch.cuda.Stream(self.device)
        # per flag word: its views and events, reused (a word is reused only
        # after the step that used it has been decided)
        self._flag_dev = [self.flags[i:i + 1] for i in range(depth + 1)]
        self._flag_hst = [self.flags_host[i:i + 1] for i in range(depth + 1)]
        self._flags_np = self.flags_host.numpy()      # the same pinned words
        self._kernels_done = [torch.cuda.Event() for _ in range(depth + 1)]
        self._flag_landed = [torch.cuda.Event() for _ in range(depth + 1)]
        self._launch_counts = {}   # (rank, row offset) -> kernel launches of a step
        self.pending = []          # launched, undecided: (buf, t, flag slot, event, grads)
        self.launched = 0          # steps launched (speculative re-runs included)
        self.kernel_launches = 0   # kernels launched (one per rank and launch window)

    def _free_buf(self, exclude):
        return next(i for i in range(self.depth + 2) if i not in exclude)

    def _launch_one(self, grads, in_buf, out_buf, t):
        slot = self.launched % (self.depth + 1)
        self.launched += 1
        flag = self._flag_dev[slot]
        self.h.step = t
        for r in self.ranks:
            key = (r, int(grads[r].offset))
            count = self._launch_counts.get(key)
            if count is None:
                count = _abi.fused_launch_count(int(self.layouts[r].length), self.bucket, key[1])
                self._launch_counts[key] = count
            self.kernel_launches += count
            st = self.state[r]
            gbuf, goff = self._gathered_target(r, out_buf)
            _abi.zero_step_shard(grads[r], self.layouts[r], st.states[in_buf],
                                 st.states[out_buf], gbuf, goff, self.bucket, self.loss_scale,
                                 self.h, flag, self.stream)
        done = self._kernels_done[slot]
        done.record(self.stream)
        self.flag_stream.wait_event(done)
        with torch.cuda.stream(self.flag_stream):
            self._flag_hst[slot].copy_(flag, non_blocking=True)
        ev = self._flag_landed[slot]         # this step's kernels and flag copy are done
        ev.record(self.flag_stream)
        self.pending.append((out_buf, t, slot, ev, grads))

    def launch(self, grads: dict) -> list:
        """Launch one step (speculating that every undecided step commits);
        decides and returns the steps that can be decided without stalling."""
        if self.pending:
            in_buf, t_in = self.pending[-1][0], self.pending[-1][1]
        else:
            in_buf, t_in = self.gcur, self.t
        out_buf = self._free_buf({self.gcur, in_buf} | {p[0] for p in self.pending})
        self._launch_one(grads, in_buf, out_buf, t_in + 1)
        decided = []
        while len(self.pending) > self.depth:
            decided.append(self._decide_oldest())
        return decided

    def _decide_oldest(self) -> bool:
        out_buf, t, slot, ev, grads = self.pending.pop(0)
        ev.synchronize()
        word = int(self._flags_np[slot])
        # every rank takes part in the decision before any rank raises
        skipped = global_skip(word != 0, self.pg, self.device)
        if word & _abi.ZERO_STEP_FLAG_WAIT_TIMEOUT:
            # a kernel's pipeline wait expired: the committed state stays, and
            # the speculative steps built on this one are dropped (their
            # kernels finish first in stream order; their flags are cleared)
            with torch.cuda.stream(self.stream):
                for s in [slot] + [p[2] for p in self.pending]:
                    self.flags[s:s + 1].zero_()
            for p in self.pending:
                p[3].synchronize()
            self.pending = []
            self.stream.synchronize()
            raise _abi.ZeroError(_abi.ZERO_ERR_TIMEOUT, "step kernel")
        self.skipped_steps.append(skipped)
        if not skipped:
            for r in self.ranks:
                self.state[r].cur = out_buf
            self.gcur = out_buf
            self.t = t
            return False
        # skipped: clear its flag word, discard the speculative steps that
        # built on it and run them again from the committed state
        with torch.cuda.stream(self.stream):
            self.flags[slot:slot + 1].zero_()
        redo = [p[4] for p in self.pending]
        for p in self.pending:
            p[3].synchronize()
            with torch.cuda.stream(self.stream):
                self.flags[p[2]:p[2] + 1].zero_()
        self.pending = []
        for g in redo:
            in_buf, t_in = (self.pending[-1][0], self.pending[-1][1]) if self.pending else \
                (self.gcur, self.t)
            out = self._free_buf({self.gcur, in_buf} | {p[0] for p in self.pending})
            self._launch_one(g, in_buf, out, t_in + 1)
        return True

    def finish(self) -> list:
        """Decide every launched step."""
        decided = []
        while self.pending:
            decided.append(self._decide_oldest())
        return decided

    def step(self, grads: dict) -> bool:
        self.launch(grads)
        return self.finish()[-1]
