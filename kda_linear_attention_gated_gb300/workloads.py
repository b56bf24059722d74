"""Seeded synthetic inputs for the KDA state update (no KDA arithmetic here).

Every tensor is drawn on the CPU from ``torch.Generator().manual_seed(seed)``
so that the CUDA path and the CPU oracle see identical bits; callers copy to
the device.  The shapes and distributions follow the workloads the method is
measured on (ROCm/ATOM pull request 2130, What and Memory: 69 KDA layers,
a [12, 128, 128] state per layer and slot, N = 64 requests; pull request 2945,
Method: 7 draft tokens + 1 under speculative decoding):

  tiny    N=1, HV=2, K=V=16, T=8 decode tokens, fp32 pool of 1 slot; q,k,v fp32
          N(0,1); a,b N(0,1); S0 N(0, 0.1^2); seed 0
  decode  N=64, HV=12, K=V=128, pool [256,12,128,128] ~ N(0, 0.1^2); q,k,v bf16
          N(0,1); a,b fp32 N(0,1); 64 distinct active slots, a seeded random
          subset (fp32 pool: seed 0; fp16 pool = fp32 draw rounded to nearest
          even: seed 1)
  verify  N=8 requests x T=8 tokens, HV=12, K=V=128, fp16 pool of 256 slots;
          fp32 inputs as in tiny; distinct init slots and 8 distinct snapshot
          slots per request (all 72 distinct); seed 2
  sweep   69 layers x N in {1,16,64,128}, own 256-slot pool per layer; slot ids
          the first N of a seeded permutation; reset ~ Bernoulli(0.05); fp32
          inputs; seed 3

"N(0, 0.1)" for the state is read as standard deviation 0.1.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import torch


@dataclass
class StepInputs:
    """CPU tensors of one call.  For decode, the token axis is absent (T = 1)."""
    pool: torch.Tensor          # [num_slots, HV, K, V] fp32 or fp16
    init_slot: torch.Tensor     # int32 [N]
    q: torch.Tensor             # [N(,T), HV, K]
    k: torch.Tensor
    v: torch.Tensor             # [N(,T), HV, V]
    a: torch.Tensor             # fp32 [N(,T), HV, K]
    b: torch.Tensor             # fp32 [N(,T), HV]
    snap_slot: torch.Tensor | None = None  # int32 [N, T] (verify only)
    reset: torch.Tensor | None = None      # uint8 [N]
    meta: dict = field(default_factory=dict)

    def to(self, device) -> "StepInputs":
        mv = lambda t: None if t is None else t.to(device)  # noqa: E731
        return StepInputs(mv(self.pool), mv(self.init_slot), mv(self.q), mv(self.k), mv(self.v),
                          mv(self.a), mv(self.b), mv(self.snap_slot), mv(self.reset), dict(self.meta))


def _randn(g, shape, dtype=torch.float32, std=1.0):
    x = torch.randn(shape, generator=g, dtype=torch.float32)
    if std != 1.0:
        x = x * std
    return x.to(dtype)


def _gate_scale(g, hv, k):
    """A layer's learned gate scale and bias: A_log = log U(1, 16) per value
    head; dt_bias = log(expm1(dt)) with dt = exp U(log 1e-3, log 1e-1) per
    (head, key channel)."""
    a_log = torch.log(1.0 + 15.0 * torch.rand((hv,), generator=g))
    lo, hi = torch.log(torch.tensor(1e-3)), torch.log(torch.tensor(1e-1))
    dt = torch.exp(lo + (hi - lo) * torch.rand((hv, k), generator=g))
    return a_log, torch.log(torch.expm1(dt))


def make_pool(g, num_slots, hv, k, v, state_dtype, std=0.1):
    """fp32 N(0, std^2), then (fp16 pool) rounded to nearest even by the dtype cast."""
    return _randn(g, (num_slots, hv, k, v), std=std).to(state_dtype)


def make_decode(n=64, hv=12, k=128, v=128, num_slots=256, state_dtype=torch.float32,
                qkv_dtype=torch.bfloat16, seed=0, reset_p=0.0, pool=True) -> StepInputs:
    """One decode token for n requests (n distinct slots of a num_slots pool)."""
    g = torch.Generator().manual_seed(seed)
    P = make_pool(g, num_slots, hv, k, v, state_dtype) if pool else None
    slots = torch.randperm(num_slots, generator=g)[:n].to(torch.int32)
    q = _randn(g, (n, hv, k), qkv_dtype)
    kk = _randn(g, (n, hv, k), qkv_dtype)
    vv = _randn(g, (n, hv, v), qkv_dtype)
    a = _randn(g, (n, hv, k))
    b = _randn(g, (n, hv))
    reset = None
    if reset_p > 0:
        reset = (torch.rand((n,), generator=g) < reset_p).to(torch.uint8)
    return StepInputs(P, slots, q, kk, vv, a, b, None, reset,
                      dict(kind="decode", n=n, hv=hv, k=k, v=v, num_slots=num_slots, seed=seed))


def make_verify(n=8, t=8, hv=12, k=128, v=128, num_slots=256, state_dtype=torch.float16,
                qkv_dtype=torch.float32, seed=2, reset_p=0.0) -> StepInputs:
    """t tokens for each of n requests; init slots and snapshot slots all distinct."""
    if n * (t + 1) > num_slots:
        raise ValueError("not enough slots for distinct init and snapshot slots")
    g = torch.Generator().manual_seed(seed)
    P = make_pool(g, num_slots, hv, k, v, state_dtype)
    perm = torch.randperm(num_slots, generator=g).to(torch.int32)
    init = perm[:n].clone()
    snap = perm[n:n + n * t].reshape(n, t).clone()
    q = _randn(g, (n, t, hv, k), qkv_dtype)
    kk = _randn(g, (n, t, hv, k), qkv_dtype)
    vv = _randn(g, (n, t, hv, v), qkv_dtype)
    a = _randn(g, (n, t, hv, k))
    b = _randn(g, (n, t, hv))
    reset = None
    if reset_p > 0:
        reset = (torch.rand((n,), generator=g) < reset_p).to(torch.uint8)
    return StepInputs(P, init, q, kk, vv, a, b, snap, reset,
                      dict(kind="verify", n=n, t=t, hv=hv, k=k, v=v, num_slots=num_slots, seed=seed))


def make_tiny(seed=0):
    """Config 'tiny': a 1-slot fp32 pool and T=8 decode tokens (returned stacked [T, ...])."""
    g = torch.Generator().manual_seed(seed)
    hv, k, v, t = 2, 16, 16, 8
    P = make_pool(g, 1, hv, k, v, torch.float32)
    q = _randn(g, (t, 1, hv, k))
    kk = _randn(g, (t, 1, hv, k))
    vv = _randn(g, (t, 1, hv, v))
    a = _randn(g, (t, 1, hv, k))
    b = _randn(g, (t, 1, hv))
    return dict(pool=P, slot=torch.zeros(1, dtype=torch.int32), q=q, k=kk, v=vv, a=a, b=b)


def make_sweep_layer(layer: int, n: int, state_dtype, hv=12, k=128, v=128, num_slots=256,
                     seed=3, reset_p=0.05, sentinel=None) -> StepInputs:
    """One layer of the 69-layer sweep.  Active slots get N(0, 0.1^2) states;
    the other slots are filled with ``sentinel`` when given (a value no update
    produces, so stray writes show), else drawn like the active ones."""
    g = torch.Generator().manual_seed(seed * 1_000_003 + layer * 1009 + n)
    perm = torch.randperm(num_slots, generator=g)
    slots = perm[:n].to(torch.int32)
    if sentinel is None:
        P = make_pool(g, num_slots, hv, k, v, state_dtype)
    else:
        P = torch.full((num_slots, hv, k, v), sentinel, dtype=state_dtype)
        P[slots.long()] = make_pool(g, n, hv, k, v, state_dtype)
    q = _randn(g, (n, hv, k))
    kk = _randn(g, (n, hv, k))
    vv = _randn(g, (n, hv, v))
    a = _randn(g, (n, hv, k))
    b = _randn(g, (n, hv))
    reset = (torch.rand((n,), generator=g) < reset_p).to(torch.uint8)
    return StepInputs(P, slots, q, kk, vv, a, b, None, reset,
                      dict(kind="decode", layer=layer, n=n, hv=hv, k=k, v=v,
                           num_slots=num_slots, seed=seed))


@dataclass
class GeneralInputs:
    """CPU tensors of one general step (packed tokens, slot table)."""
    pool: torch.Tensor                 # [num_slots, HV, K, V] fp32 or fp16
    slot_table: torch.Tensor           # int32 [N, C]
    q: torch.Tensor                    # [total, H, K]
    k: torch.Tensor
    v: torch.Tensor                    # [total, HV, V]
    a: torch.Tensor                    # fp32 [total, HV, K]
    b: torch.Tensor                    # fp32 [total, HV]
    cu_seqlens: torch.Tensor | None = None   # int32 [N + 1]
    accepted: torch.Tensor | None = None     # int32 [N], in 1 .. C
    reset: torch.Tensor | None = None        # uint8 [N]
    a_log: torch.Tensor | None = None        # fp32 [HV]
    dt_bias: torch.Tensor | None = None      # fp32 [HV, K]
    in_place: bool = False
    max_t: int = 0
    meta: dict = field(default_factory=dict)

    def to(self, device) -> "GeneralInputs":
        mv = lambda t: None if t is None else t.to(device)  # noqa: E731
        return GeneralInputs(mv(self.pool), mv(self.slot_table), mv(self.q), mv(self.k), mv(self.v),
                             mv(self.a), mv(self.b), mv(self.cu_seqlens), mv(self.accepted), mv(self.reset),
                             mv(self.a_log), mv(self.dt_bias), self.in_place, self.max_t, dict(self.meta))


def make_general(n=8, t_lens=None, t=8, num_cols=None, h_qk=None, hv=12, k=128, v=128, num_slots=256,
                 state_dtype=torch.float16, qkv_dtype=torch.float32, seed=4, reset_p=0.0, pad_p=0.0,
                 drop_p=0.0, accepted=True, gate_scale=False, in_place=False) -> GeneralInputs:
    """A general step: requests of t_lens[r] tokens (packed; None: t each),
    a slot table of num_cols distinct slots per request, the initial column
    accepted[r] - 1 drawn uniformly, padding requests (whole row -1) with
    probability pad_p, kept-snapshot entries dropped (-1) with probability
    drop_p (never the initial column), grouped q/k heads (h_qk), and the
    learned gate scale (A_log = log U(1, 16), dt_bias = log(expm1(dt)),
    dt = exp U(log 1e-3, log 1e-1)).  in_place: one token per request, stored
    back to the initial slot."""
    g = torch.Generator().manual_seed(seed)
    h_qk = hv if h_qk is None else h_qk
    if in_place:
        t_lens, t = None, 1
    lens = [t] * n if t_lens is None else list(t_lens)
    max_t = max(lens) if lens else 0
    num_cols = max(max_t, 1) if num_cols is None else num_cols
    if n * num_cols > num_slots:
        raise ValueError("not enough slots for a table of distinct slots")
    P = make_pool(g, num_slots, hv, k, v, state_dtype)
    table = torch.randperm(num_slots, generator=g)[:n * num_cols].to(torch.int32).reshape(n, num_cols).clone()
    total = sum(lens)
    q = _randn(g, (total, h_qk, k), qkv_dtype)
    kk = _randn(g, (total, h_qk, k), qkv_dtype)
    vv = _randn(g, (total, hv, v), qkv_dtype)
    a = _randn(g, (total, hv, k))
    b = _randn(g, (total, hv))
    acc = None
    if accepted:
        acc = (torch.randint(0, num_cols, (n,), generator=g) + 1).to(torch.int32)
    c0 = acc.long() - 1 if acc is not None else torch.zeros(n, dtype=torch.long)
    if drop_p > 0:
        drop = torch.rand((n, num_cols), generator=g) < drop_p
        drop[torch.arange(n), c0] = False
        table[drop] = -1
    if pad_p > 0:
        pad = torch.rand((n,), generator=g) < pad_p
        table[pad] = -1
    reset = None
    if reset_p > 0:
        reset = (torch.rand((n,), generator=g) < reset_p).to(torch.uint8)
    a_log, dt_bias = _gate_scale(g, hv, k) if gate_scale else (None, None)
    cu = None
    if t_lens is not None:
        cu = torch.zeros(n + 1, dtype=torch.int32)
        cu[1:] = torch.cumsum(torch.tensor(lens, dtype=torch.int64), 0).to(torch.int32)
    return GeneralInputs(P, table, q, kk, vv, a, b, cu, acc, reset, a_log, dt_bias, in_place, max_t,
                         dict(kind="general", n=n, hv=hv, h_qk=h_qk, k=k, v=v, num_slots=num_slots,
                              seed=seed, lens=lens))


@dataclass
class ConvInputs:
    """CPU tensors of one causal short-convolution step with its paged window."""
    window: torch.Tensor               # [num_slots, L, C] fp32, fp16 or bf16
    conv_slot: torch.Tensor            # int32 [N]
    x: torch.Tensor                    # [total, C], the window's dtype
    weight: torch.Tensor               # fp32 [C, KW]
    bias: torch.Tensor | None = None   # fp32 [C]
    cu_seqlens: torch.Tensor | None = None
    accepted: torch.Tensor | None = None  # int32 [N], 1 .. L - KW + 2
    reset: torch.Tensor | None = None
    max_t: int = 0
    meta: dict = field(default_factory=dict)

    def to(self, device) -> "ConvInputs":
        mv = lambda t: None if t is None else t.to(device)  # noqa: E731
        return ConvInputs(mv(self.window), mv(self.conv_slot), mv(self.x), mv(self.weight), mv(self.bias),
                          mv(self.cu_seqlens), mv(self.accepted), mv(self.reset), self.max_t, dict(self.meta))


def make_conv(n=8, t=5, t_lens=None, channels=4608, kw=4, num_spec=4, num_slots=64, dtype=torch.bfloat16,
              seed=5, accepted=True, reset_p=0.0, pad_p=0.0, bias=True) -> ConvInputs:
    """The short convolution in front of the recurrence: window length
    L = kw - 1 + num_spec (the conv pool's kernel - 1 + num_spec), qlen =
    num_spec + 1 tokens per request (or t_lens), channels = 2 * 12 * 128 +
    12 * 128 by default (q, k and v of one layer); window and x ~ N(0, 1) in
    dtype, weight ~ N(0, 1 / kw), bias ~ N(0, 0.1^2); accepted[r] uniform in
    1 .. num_spec + 1."""
    g = torch.Generator().manual_seed(seed)
    L = kw - 1 + num_spec
    lens = [t] * n if t_lens is None else list(t_lens)
    total = sum(lens)
    W = _randn(g, (num_slots, L, channels), dtype)
    slots = torch.randperm(num_slots, generator=g)[:n].to(torch.int32)
    x = _randn(g, (total, channels), dtype)
    w = _randn(g, (channels, kw), std=1.0 / kw ** 0.5)
    b = _randn(g, (channels,), std=0.1) if bias else None
    acc = (torch.randint(0, num_spec + 1, (n,), generator=g) + 1).to(torch.int32) if accepted else None
    if pad_p > 0:
        slots[torch.rand((n,), generator=g) < pad_p] = -1
    reset = (torch.rand((n,), generator=g) < reset_p).to(torch.uint8) if reset_p > 0 else None
    cu = None
    if t_lens is not None:
        cu = torch.zeros(n + 1, dtype=torch.int32)
        cu[1:] = torch.cumsum(torch.tensor(lens, dtype=torch.int64), 0).to(torch.int32)
    return ConvInputs(W, slots, x, w, b, cu, acc, reset, max(lens) if lens else 0,
                      dict(kind="conv", n=n, kw=kw, L=L, channels=channels, seed=seed, lens=lens))


@dataclass
class DecodeConvInputs:
    """CPU tensors of one decode step with the short convolution fused in front."""
    pool: torch.Tensor                 # [num_slots, HV, K, V] fp32 or fp16
    slot_ids: torch.Tensor             # int32 [N]
    window: torch.Tensor               # [num_wslots, L, C] fp32, fp16 or bf16
    conv_slot: torch.Tensor            # int32 [N]
    x: torch.Tensor                    # [N, C] of the window's dtype: q | k | v channels
    weight: torch.Tensor               # fp32 [C, KW]
    bias: torch.Tensor | None          # fp32 [C]
    a: torch.Tensor                    # fp32 [N, HV, K]
    b: torch.Tensor                    # fp32 [N, HV]
    reset: torch.Tensor | None = None  # uint8 [N]
    h_qk: int = 12
    meta: dict = field(default_factory=dict)
    a_log: torch.Tensor | None = None    # fp32 [HV]
    dt_bias: torch.Tensor | None = None  # fp32 [HV, K]

    def to(self, device) -> "DecodeConvInputs":
        mv = lambda t: None if t is None else t.to(device)  # noqa: E731
        return DecodeConvInputs(mv(self.pool), mv(self.slot_ids), mv(self.window), mv(self.conv_slot), mv(self.x),
                                mv(self.weight), mv(self.bias), mv(self.a), mv(self.b), mv(self.reset), self.h_qk,
                                dict(self.meta), mv(self.a_log), mv(self.dt_bias))


def make_decode_conv(n=64, hv=12, h_qk=12, k=128, v=128, kw=4, L=3, num_slots=256, num_wslots=256,
                     state_dtype=torch.float32, dtype=torch.bfloat16, seed=11, reset_p=0.0,
                     bias=True, gate_scale=False) -> DecodeConvInputs:
    """One decode token for n requests with the short convolution in front:
    channels C = 2 h_qk k + hv v; the state pool as in make_decode; the window
    (L entries) and x ~ N(0, 1) in dtype, weight ~ N(0, 1 / kw), bias ~
    N(0, 0.1^2), as in make_conv; a, b ~ N(0, 1); n distinct state slots and
    n distinct window slots; gate_scale: the learned gate scale and bias as in
    make_general."""
    g = torch.Generator().manual_seed(seed)
    C = 2 * h_qk * k + hv * v
    P = make_pool(g, num_slots, hv, k, v, state_dtype)
    slots = torch.randperm(num_slots, generator=g)[:n].to(torch.int32)
    W = _randn(g, (num_wslots, L, C), dtype)
    cslots = torch.randperm(num_wslots, generator=g)[:n].to(torch.int32)
    x = _randn(g, (n, C), dtype)
    w = _randn(g, (C, kw), std=1.0 / kw ** 0.5)
    bv = _randn(g, (C,), std=0.1) if bias else None
    a = _randn(g, (n, hv, k))
    b = _randn(g, (n, hv))
    reset = (torch.rand((n,), generator=g) < reset_p).to(torch.uint8) if reset_p > 0 else None
    a_log, dt_bias = _gate_scale(g, hv, k) if gate_scale else (None, None)
    return DecodeConvInputs(P, slots, W, cslots, x, w, bv, a, b, reset, h_qk,
                            dict(kind="decode_conv", n=n, hv=hv, h_qk=h_qk, k=k, v=v, kw=kw, L=L, seed=seed),
                            a_log, dt_bias)


@dataclass
class StepConvInputs:
    """CPU tensors of one speculative step with the short convolution fused in front."""
    pool: torch.Tensor                 # [num_slots, HV, K, V]
    slot_table: torch.Tensor           # int32 [N, num_cols] (a padding request's row is -1)
    accepted: torch.Tensor             # int32 [N]
    cu_seqlens: torch.Tensor | None    # int32 [N + 1] or None
    max_t: int
    window: torch.Tensor               # [num_wslots, L, C]
    conv_slot: torch.Tensor            # int32 [N] (-1 for a padding request)
    x: torch.Tensor                    # [total, C]: q | k | v channels
    weight: torch.Tensor               # fp32 [C, KW]
    bias: torch.Tensor | None
    a: torch.Tensor                    # fp32 [total, HV, K]
    b: torch.Tensor                    # fp32 [total, HV]
    reset: torch.Tensor | None = None
    a_log: torch.Tensor | None = None
    dt_bias: torch.Tensor | None = None
    h_qk: int = 12
    meta: dict = field(default_factory=dict)

    def to(self, device) -> "StepConvInputs":
        mv = lambda t: None if t is None else t.to(device)  # noqa: E731
        return StepConvInputs(mv(self.pool), mv(self.slot_table), mv(self.accepted), mv(self.cu_seqlens), self.max_t,
                              mv(self.window), mv(self.conv_slot), mv(self.x), mv(self.weight), mv(self.bias),
                              mv(self.a), mv(self.b), mv(self.reset), mv(self.a_log), mv(self.dt_bias), self.h_qk,
                              dict(self.meta))


def make_step_conv(n=8, num_spec=4, t_lens=None, h_qk=12, hv=12, k=128, v=128, kw=4, num_slots=256, num_wslots=64,
                   state_dtype=torch.float16, dtype=torch.bfloat16, seed=60, reset_p=0.0, pad_p=0.0,
                   gate_scale=False, bias=True) -> StepConvInputs:
    """A speculative step of n requests (num_spec + 1 tokens each, or t_lens)
    with the conv window in front: L = kw - 1 + num_spec entries, a slot table
    of num_spec + 1 distinct slots per request; accepted[r] drawn uniformly
    among the values a request of T_r tokens admits (the window keeps
    L - T_r old entries, which must lie below acc + kw - 1): max(1, num_spec -
    T_r + 1) .. num_spec + 1.  Window, x ~ N(0, 1) in dtype, weight ~
    N(0, 1 / kw), bias ~ N(0, 0.1^2) as in make_conv; the pool, a, b as in
    make_general; padding requests (probability pad_p) have a slot-table row
    and a window slot of -1."""
    g = torch.Generator().manual_seed(seed)
    L = kw - 1 + num_spec
    ncols = num_spec + 1
    lens = [ncols] * n if t_lens is None else list(t_lens)
    if max(lens) > ncols:
        raise ValueError("a request has more tokens than num_spec + 1")
    total = sum(lens)
    C = 2 * h_qk * k + hv * v
    P = make_pool(g, num_slots, hv, k, v, state_dtype)
    table = torch.randperm(num_slots, generator=g)[:n * ncols].to(torch.int32).reshape(n, ncols).clone()
    acc = torch.tensor([int(torch.randint(max(1, num_spec - t + 1), ncols + 1, (1,), generator=g)) for t in lens],
                       dtype=torch.int32)
    W = _randn(g, (num_wslots, L, C), dtype)
    cslots = torch.randperm(num_wslots, generator=g)[:n].to(torch.int32)
    x = _randn(g, (total, C), dtype)
    w = _randn(g, (C, kw), std=1.0 / kw ** 0.5)
    bv = _randn(g, (C,), std=0.1) if bias else None
    a = _randn(g, (total, hv, k))
    b = _randn(g, (total, hv))
    reset = (torch.rand((n,), generator=g) < reset_p).to(torch.uint8) if reset_p > 0 else None
    if pad_p > 0:
        pad = torch.rand((n,), generator=g) < pad_p
        table[pad] = -1
        cslots[pad] = -1
    a_log, dt_bias = _gate_scale(g, hv, k) if gate_scale else (None, None)
    cu = None
    if t_lens is not None:
        cu = torch.zeros(n + 1, dtype=torch.int32)
        cu[1:] = torch.cumsum(torch.tensor(lens, dtype=torch.int64), 0).to(torch.int32)
    return StepConvInputs(P, table, acc, cu, max(lens), W, cslots, x, w, bv, a, b, reset, a_log, dt_bias, h_qk,
                          dict(kind="step_conv", n=n, num_spec=num_spec, lens=lens, kw=kw, L=L, seed=seed))


@dataclass
class PrefillInputs:
    """CPU tensors of one prefill call over packed prompts."""
    pool: torch.Tensor
    init_slot: torch.Tensor            # int32 [N]
    final_slot: torch.Tensor           # int32 [N]
    q: torch.Tensor                    # [total, H, K]
    k: torch.Tensor
    v: torch.Tensor                    # [total, HV, V]
    a: torch.Tensor                    # fp32 [total, HV, K]
    b: torch.Tensor                    # fp32 [total, HV]
    cu_seqlens: torch.Tensor | None = None
    reset: torch.Tensor | None = None
    a_log: torch.Tensor | None = None
    dt_bias: torch.Tensor | None = None
    max_t: int = 0
    meta: dict = field(default_factory=dict)

    def to(self, device) -> "PrefillInputs":
        mv = lambda t: None if t is None else t.to(device)  # noqa: E731
        return PrefillInputs(mv(self.pool), mv(self.init_slot), mv(self.final_slot), mv(self.q), mv(self.k),
                             mv(self.v), mv(self.a), mv(self.b), mv(self.cu_seqlens), mv(self.reset),
                             mv(self.a_log), mv(self.dt_bias), self.max_t, dict(self.meta))


def make_prefill(lens=(200, 37), h_qk=None, hv=12, k=128, v=128, num_slots=16, state_dtype=torch.float16,
                 qkv_dtype=torch.bfloat16, seed=6, reset_p=0.5, same_slot_p=0.5, gate_scale=False,
                 pad_p=0.0) -> PrefillInputs:
    """Prompts of the given lengths (packed; cu_seqlens always given), q/k/v
    N(0, 1) in qkv_dtype, a, b N(0, 1); a request starts from zero (fresh
    prompt, probability reset_p) or from a slot's state, and its final state
    goes to its own slot or to a fresh one.  The gate-scale draws follow
    make_general."""
    g = torch.Generator().manual_seed(seed)
    n = len(lens)
    h_qk = hv if h_qk is None else h_qk
    if 2 * n > num_slots:
        raise ValueError("not enough slots")
    P = make_pool(g, num_slots, hv, k, v, state_dtype)
    perm = torch.randperm(num_slots, generator=g).to(torch.int32)
    init = perm[:n].clone()
    final = torch.where(torch.rand((n,), generator=g) < same_slot_p, init, perm[n:2 * n])
    total = int(sum(lens))
    q = _randn(g, (total, h_qk, k), qkv_dtype)
    kk = _randn(g, (total, h_qk, k), qkv_dtype)
    vv = _randn(g, (total, hv, v), qkv_dtype)
    a = _randn(g, (total, hv, k))
    b = _randn(g, (total, hv))
    reset = (torch.rand((n,), generator=g) < reset_p).to(torch.uint8)
    if pad_p > 0:
        init[torch.rand((n,), generator=g) < pad_p] = -1
    a_log = dt_bias = None
    if gate_scale:
        a_log = torch.log(1.0 + 15.0 * torch.rand((hv,), generator=g))
        lo, hi = torch.log(torch.tensor(1e-3)), torch.log(torch.tensor(1e-1))
        dt_bias = torch.log(torch.expm1(torch.exp(lo + (hi - lo) * torch.rand((hv, k), generator=g))))
    cu = torch.zeros(n + 1, dtype=torch.int32)
    cu[1:] = torch.cumsum(torch.tensor(list(lens), dtype=torch.int64), 0).to(torch.int32)
    return PrefillInputs(P, init, final.to(torch.int32), q, kk, vv, a, b, cu, reset, a_log, dt_bias,
                         max(lens) if lens else 0, dict(kind="prefill", lens=list(lens), seed=seed))
