"""Temporal chunk parallelism: one video split along time over ranks, with the causal halo exchange.

"SwiftVR Inference Optimization" (LightX2V blog), sections "Scaling Across GPUs Along the Time
Axis" and "ReAE: Causal Halo Exchange": every rank holds the whole layer stack and owns a
contiguous range of frames.  A causal layer with temporal extent kt needs, for the first frame of
a rank's range, the layer's *input* features of the kt - 1 frames before it.  Those belong to the
preceding rank, and they are known as soon as that rank has the layer's input, so before each
causal layer every rank sends the last kt - 1 input frames of its range to the next rank and
receives its own history from the previous one; then all ranks compute the layer at once.  The
video's first frames take a zero history.  When the video is processed in waves of `world`
chunks, rank 0 keeps the boundary that the last rank of one wave sends back for the first chunk of
the next wave.  ("SGLang-Diffusion advanced optimizations", section 3 "Parallel VAE": splitting
the VAE's convolutions with a halo exchange keeps the result equal to the unsplit one.)

Because the library's result does not depend on how a video is cut into chunks (every output is
accumulated in the same order), the time-split result equals the one-device result bit for bit.

The exchange is point-to-point (torch.distributed isend / irecv: NCCL for device tensors, gloo for
host tensors) into buffers the receiving rank owns; no reduction, no peer loads.  The boundary a
rank sends is the last kt - 1 frames of concat(history, input), so a rank holding fewer than
kt - 1 frames first waits for its own history, then sends; rank 0 never waits, so the chain ends.

    layers = [ChunkedLayer(plan1, w1, b1), ChunkedLayer(plan2, w2, b2)]
    split = TimeSplit(layers)                 # inside an initialised process group
    y_local = split.forward(x_local)          # this rank's frames of one wave

The height split ("SGLang-Diffusion advanced optimizations", section 3 "Parallel VAE": every rank
takes a band of rows, exchanges halo rows with its neighbours, and the bands are gathered at the
end): every rank owns a contiguous band of rows of every frame and runs each layer on its band
extended by the (kh - 1) / 2 rows above and below that its neighbours send it.  The outputs of the
band's own rows equal the whole frame's (the rows outside the frame are the conv's zero padding,
the rows from the neighbours are the real ones); the extended rows' outputs are dropped.  Each
rank keeps its layers' temporal histories itself (of its extended band, halo rows included).

    split = HeightSplit([ChunkedLayer(plan_band1, w1, b1), ...])   # plans of the extended band
    y_band = split.forward(x_band)            # one chunk of this rank's rows
    y = split.gather(y_band, H)               # every rank's bands, whole frames
"""
from __future__ import annotations

__all__ = ["frame_ranges", "end_history", "exchange", "TimeSplit", "ChunkedLayer", "row_ranges",
           "band_extent", "HeightSplit"]


def frame_ranges(T: int, world: int):
    """Contiguous frame ranges [(start, stop)] of a T-frame video over `world` ranks, the first
    T % world ranks one frame longer."""
    if T < 0 or world < 1:
        raise ValueError("T >= 0 and world >= 1 required")
    base, extra = divmod(T, world)
    out, s = [], 0
    for r in range(world):
        n = base + (1 if r < extra else 0)
        out.append((s, s + n))
        s += n
    return out


def end_history(history, x, P: int):
    """The last P frames of concat(history, x): the history the frames after x need (history has
    P frames; for a range of at least P frames it is the range's last P frames)."""
    import torch
    T = int(x.shape[0])
    if T >= P:
        return x[T - P:]
    return torch.cat([history[T:], x], 0)


def exchange(x_local, P: int, out=None, group=None):
    """One layer's halo exchange without waves: every rank sends the last P frames of its range to
    the next rank and returns the P frames it received from the previous one (rank 0: zeros).
    Each range must hold at least P frames.  `out` ([P, ...], like a frame of x_local) receives
    the history when given.  Device tensors go through NCCL, ordered on the current stream."""
    import torch
    import torch.distributed as dist
    rank, world = _group_info(group)
    if int(x_local.shape[0]) < P:
        raise ValueError("exchange needs at least P frames per rank")
    shape = (P,) + tuple(x_local.shape[1:])
    hist = out if out is not None else torch.empty(shape, dtype=x_local.dtype, device=x_local.device)
    if P == 0:
        return hist
    reqs = []
    if rank == 0:
        hist.zero_()
    else:
        reqs.append(dist.irecv(hist, src=_global_rank(group, rank - 1), group=group))
    if rank < world - 1:
        reqs.append(dist.isend(x_local[int(x_local.shape[0]) - P:], dst=_global_rank(group, rank + 1), group=group))
    for r in reqs:
        r.wait()
    return hist


def _group_info(group):
    import torch.distributed as dist
    if not dist.is_available() or not dist.is_initialized():
        return 0, 1
    return dist.get_rank(group), dist.get_world_size(group)


def _global_rank(group, r):
    import torch.distributed as dist
    return r if group is None else dist.get_global_rank(group, r)


class TimeSplit:
    """A stack of causal layers run on this rank's frames, with the halo exchange before every
    layer that has a history.  Each layer is a callable (x_local, history) -> y_local with an
    attribute P = kt - 1 (history=None means a zero history; P = 0 layers get None).  Successive
    forward calls are successive waves: rank 0 starts a wave from the boundary the last rank sent
    at the end of the previous one (zeros for the first wave)."""

    def __init__(self, layers, group=None):
        self.layers = list(layers)
        self.group = group
        self._carry = [None] * len(self.layers)
        self.last_histories = []  # the history each layer received in the latest forward

    def reset(self):
        """Start a new video: the next wave's first chunk takes a zero history again."""
        self._carry = [None] * len(self.layers)

    def forward(self, x_local):
        import torch
        import torch.distributed as dist
        rank, world = _group_info(self.group)
        nxt, prv = _global_rank(self.group, (rank + 1) % world), _global_rank(self.group, (rank - 1) % world)
        first = _global_rank(self.group, 0)
        pending = []  # (request, tensor kept alive until the request completes)
        wrap_in = []  # rank 0: (layer, buffer, request) of the boundaries the last rank sends back
        self.last_histories = []
        x = x_local
        for i, layer in enumerate(self.layers):
            P = int(layer.P)
            if P == 0:
                self.last_histories.append(None)
                x = layer(x, None)
                continue
            shape = (P,) + tuple(x.shape[1:])
            recv = None
            if rank == 0:
                hist = self._carry[i]
                if hist is None:
                    hist = torch.zeros(shape, dtype=x.dtype, device=x.device)
            else:
                hist = torch.empty(shape, dtype=x.dtype, device=x.device)
                recv = dist.irecv(hist, src=prv, group=self.group, tag=2 * i)
            if int(x.shape[0]) < P and recv is not None:
                recv.wait()  # the boundary to send includes part of this rank's own history
                recv = None
            end = end_history(hist, x, P).contiguous()
            if rank < world - 1:
                pending.append((dist.isend(end, dst=nxt, group=self.group, tag=2 * i), end))
            elif world == 1:
                self._carry[i] = end.clone()
            else:
                pending.append((dist.isend(end, dst=first, group=self.group, tag=2 * i + 1), end))
            if rank == 0 and world > 1:
                buf = torch.empty(shape, dtype=x.dtype, device=x.device)
                wrap_in.append((i, buf, dist.irecv(buf, src=_global_rank(self.group, world - 1), group=self.group,
                                                   tag=2 * i + 1)))
            if recv is not None:
                recv.wait()
            self.last_histories.append(hist)
            x = layer(x, hist)
        for i, buf, req in wrap_in:
            req.wait()
            self._carry[i] = buf
        for req, _ in pending:
            req.wait()
        return x


def row_ranges(H: int, world: int):
    """Contiguous row bands [(start, stop)] of H-row frames over `world` ranks (as frame_ranges)."""
    return frame_ranges(H, world)


def band_extent(H: int, world: int, rank: int, halo: int):
    """(first, stop) rows of rank's band extended by `halo` rows on each side that lies inside
    the frame: the rows a layer with a (2 * halo + 1)-row spatial kernel reads for the band."""
    a, b = row_ranges(H, world)[rank]
    return max(0, a - halo), min(H, b + halo)


class HeightSplit:
    """A stack of layers run on this rank's band of rows, with the halo-row exchange before every
    layer.  Each layer is a callable (x_extended, history) -> y_extended with attributes P (= kt - 1)
    and halo (= (kh - 1) / 2); it is run on the band extended by up to `halo` rows above and below
    (the neighbours' rows; none beyond the frame's edge) and must be built for that height (see
    band_extent).  The layer's temporal history (of the extended band) stays on the rank: the
    history a layer returns through its attribute `last_history` after a call is passed back to it
    on the next chunk (None: zero history, the first chunk of a video)."""

    def __init__(self, layers, group=None):
        self.layers = list(layers)
        self.group = group
        self.histories = [None] * len(self.layers)

    def reset(self):
        self.histories = [None] * len(self.layers)

    def _extend(self, x, halo, rank, world):
        """x [T][h][W][C] (this rank's band) -> the band with `halo` neighbour rows on each side
        that has a neighbour, and the number of rows added on top."""
        import torch
        import torch.distributed as dist
        if halo == 0 or world == 1:
            return x, 0
        if int(x.shape[1]) < halo:
            raise ValueError("every band needs at least the halo's rows")
        up, down = _global_rank(self.group, rank - 1), _global_rank(self.group, rank + 1)
        reqs, keep = [], []
        top = bottom = None
        shape = (x.shape[0], halo) + tuple(x.shape[2:])
        if rank > 0:
            top = torch.empty(shape, dtype=x.dtype, device=x.device)
            reqs.append(dist.irecv(top, src=up, group=self.group, tag=1))
            first = x[:, :halo].contiguous()
            keep.append(first)
            reqs.append(dist.isend(first, dst=up, group=self.group, tag=2))
        if rank < world - 1:
            bottom = torch.empty(shape, dtype=x.dtype, device=x.device)
            reqs.append(dist.irecv(bottom, src=down, group=self.group, tag=2))
            last = x[:, int(x.shape[1]) - halo:].contiguous()
            keep.append(last)
            reqs.append(dist.isend(last, dst=down, group=self.group, tag=1))
        for r in reqs:
            r.wait()
        parts = [p for p in (top, x, bottom) if p is not None]
        return torch.cat(parts, 1), (halo if top is not None else 0)

    def forward(self, x_band):
        rank, world = _group_info(self.group)
        x = x_band
        for i, layer in enumerate(self.layers):
            halo = int(getattr(layer, "halo", 0))
            xe, top = self._extend(x, halo, rank, world)
            y = layer(xe, self.histories[i] if int(layer.P) > 0 else None)
            if int(layer.P) > 0:
                self.histories[i] = layer.last_history
            x = y[:, top:top + int(x.shape[1])]
        return x

    def gather(self, y_band, H: int):
        """Every rank's band of the output, whole frames [T][H][W][C], on every rank."""
        import torch
        import torch.distributed as dist
        rank, world = _group_info(self.group)
        if world == 1:
            return y_band
        ranges = row_ranges(H, world)
        hmax = max(b - a for a, b in ranges)
        pad = torch.zeros((y_band.shape[0], hmax) + tuple(y_band.shape[2:]), dtype=y_band.dtype,
                          device=y_band.device)
        pad[:, :int(y_band.shape[1])] = y_band
        bufs = [torch.empty_like(pad) for _ in range(world)]
        dist.all_gather(bufs, pad, group=self.group)
        return torch.cat([bufs[r][:, :b - a] for r, (a, b) in enumerate(ranges)], 1)


class ChunkedLayer:
    """One layer of the library run over a rank's frames: the chunk loop with the two ping-pong
    history buffers, the first chunk reading the history the exchange delivered.  plan is a
    CausalConv3dPlan (or Upsample2xConvPlan), w / b / residual its tensors."""

    def __init__(self, plan, w, b=None, chunk: int = 4, stream=None):
        if chunk < 1:
            raise ValueError("chunk >= 1")
        self.plan, self.w, self.b, self.chunk, self.stream = plan, w, b, int(chunk), stream
        self.P = plan.kt - 1
        self.halo = (plan.kh - 1) // 2
        self._caches = None
        self.last_history = None  # the history the last call left (the input frames after it need)

    def __call__(self, x, history, residual=None):
        import torch
        T = int(x.shape[0])
        y = torch.empty((T, self.plan.Ho, self.plan.Wo, self.plan.Cout), dtype=self.plan.torch_dtype(),
                        device=x.device)
        if self.P > 0 and self._caches is None:
            # three buffers: the two the chunks alternate between, and a third so that neither of
            # them is the history passed in (which may be the one the previous call left)
            self._caches = [self.plan.new_cache(x.device) for _ in range(3)]
        if self.P > 0:
            free = [c for c in self._caches if history is None or c.data_ptr() != history.data_ptr()][:2]
        s, k = 0, 0
        while s < T:
            c = min(self.chunk, T - s)
            if self.P > 0:
                cin = history if k == 0 else free[(k - 1) % 2]
                cout = free[k % 2]
                self.last_history = cout
            else:
                cin = cout = None
            self.plan.forward_chunk(x[s:s + c], self.w, self.b, None if residual is None else residual[s:s + c],
                                    cin, cout, y[s:s + c], stream=self.stream)
            s += c
            k += 1
        return y
