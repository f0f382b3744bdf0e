"""Host-side tests of the C ABI: the library loads and exports every symbol
the header declares, the planner partitions lists correctly, validation
rejects bad arguments.  No GPU needed (no compute call is made)."""
import ctypes
import os
import re

import numpy as np
import pytest

import oracle
from adamw_optimizer_step_sm_gb300 import adamw_sm as A
from adamw_optimizer_step_sm_gb300 import build as B

HEADER_DIR = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include")


def _declared_functions():
    names = set()
    for f in os.listdir(HEADER_DIR):
        if f.endswith(".h"):
            src = open(os.path.join(HEADER_DIR, f)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names |= set(re.findall(r"^\s*(?:const\s+)?[\w\*\s]+?\b(adamw_\w+)\s*\(", src, re.M))
    return sorted(names)


def test_library_exports_every_declared_symbol():
    lib = ctypes.CDLL(B.build())
    names = _declared_functions()
    assert "adamw_step" in names and "adamw_plan_create" in names
    missing = [n for n in names if not hasattr(lib, n)]
    assert not missing, f"declared but not exported: {missing}"


ELEM_SIZES = {0: (2, 2, 2, 2, 2), 1: (4, 2, 4, 4, 2), 2: (2, 2, 4, 4, 2), 3: (2, 2, 2, 2, 0),
              4: (2, 2, 2, 4, 2)}
# any-precision modes: bf16 param and grad; the flags make m, v, c fp32 or
# drop c (written out from the header's table, not from the library)
for _f in range(16):
    if (_f & 12) != 12:
        ELEM_SIZES[16 + _f] = (2, 2, 4 if _f & 1 else 2, 4 if _f & 2 else 2,
                               0 if _f & 8 else (4 if _f & 4 else 2))


def _fake(base, n, mode=0, skew=(0, 0, 0, 0, 0)):
    es = ELEM_SIZES[mode]
    return tuple(base + (k + 1) * (1 << 36) + s * e for k, (s, e) in enumerate(zip(skew, es))) + (n,)


def _check_partition(entries, mode, grid):
    chunks = A.adamw_plan_chunks(entries, mode, grid)
    es = ELEM_SIZES[mode]
    covered = {k: np.zeros(e[5], np.int32) for k, e in enumerate(entries)}
    per_cta = np.zeros(grid, np.int64)
    last_cta = 0
    claimable = 0
    for c in chunks:
        # every CTA's own chunks in CTA order, then the claimable ones (-1)
        if c.cta < 0:
            assert c.cta == -1 and c.len <= 8192, "claimable piece"
            last_cta = grid
            claimable += c.len
        else:
            assert c.cta < grid and c.cta >= last_cta, "chunks not in CTA order"
            last_cta = c.cta
            per_cta[c.cta] += c.len
        covered[c.tensor][c.offset:c.offset + c.len] += 1
        if c.vec:
            e = entries[c.tensor]
            for s in range(5):
                assert (e[s] + c.offset * es[s]) % 16 == 0, "vector chunk start not 16-B aligned"
    for k, cov in covered.items():
        assert np.all(cov == 1), f"tensor {k}: elements covered {set(cov.tolist())} times"
    total = sum(e[5] for e in entries)
    if total:
        # contiguous ranges: within a vector of the mean; round-robin tiles:
        # within one tile of it (the claimable last round on top, shared)
        longest = max(c.len for c in chunks)
        assert per_cta.max() <= -(-total // grid) + min(longest, total) + 4096 // max(1, grid - 1) + 16, \
            "CTA load imbalance"
        if grid > 1:
            # CTA 0's share is 4096 elements short of the others' (never
            # below zero): the device step's CTA 0 computes the next step's
            # scalars first
            others = (total - claimable - per_cta[0]) / (grid - 1)
            assert per_cta[0] <= max(0.0, others - 4096) + min(longest, total) + 16, (per_cta[0], others)
        assert claimable <= 0.55 * total, "claimable share"
        k = round(total / (grid * 8192))
        if k < 8:
            # short lists: every tile dealt
            assert claimable == 0, (claimable, k)
        if claimable:
            # the last ceil(12 % of k) rounds, k rounds of about 8192 each
            rounds = min(max(1, -(-k * 12 // 100)), k - 1)
            assert abs(claimable - total * rounds / k) <= grid * 2048 + 8192 * len(entries) + total / k, \
                (claimable, total * rounds / k)
    return chunks


def test_partition_covers_each_element_once_and_balances():
    sizes = [1, 7, 8, 9, 4095, 65537, 0, 3, 1000003, 255, 256, 257]
    for mode in (0, 1, 2):
        entries = [_fake(i << 30, n, mode) for i, n in enumerate(sizes)]
        for grid in (1, 2, 5, 152, 608, 5000):
            _check_partition(entries, mode, grid)


@pytest.mark.parametrize("total,grid,cta0", [
    (1_048_576, 456, 0),                        # contiguous, even share 2300 < 4096: none
    (4_000_000, 456, 8776 - 4096),              # contiguous, share 8776 (vector-rounded)
    (13_850_000, 304, None),                    # round-robin tiles, 6 rounds
    (1_000, 1, 1_000)])                         # one CTA takes everything
def test_cta0_share_is_short_by_the_memo_relief(total, grid, cta0):
    """CTA 0 of the update partition gets 4096 elements less than the others
    (none when its share is smaller), so that the device step's CTA 0 can
    compute the next step's scalars first; the other CTAs stay balanced."""
    chunks = _check_partition([_fake(0, total, 0)], 0, grid)
    load = np.zeros(grid, np.int64)
    for c in chunks:
        if c.cta >= 0:
            load[c.cta] += c.len
    if cta0 is not None:
        assert load[0] == cta0, (load[0], cta0)
    if grid > 1:
        rest = load[1:]
        assert rest.max() - rest.min() <= 2048, (rest.min(), rest.max())
        if cta0 is None:
            assert abs(rest.mean() - load[0] - 4096) <= 512, (load[0], rest.mean())


@pytest.mark.parametrize("sizes,grid", [([13_850_000], 304), ([13_850_000], 456),
                                        ([125_000_007, 3, 9, 1 << 20], 456),
                                        ([1000003] * 40 + [7, 65537], 152),
                                        ([1_315_758_080], 456)])
def test_interleaved_tiles_cut_on_4k_boundaries_and_balance(sizes, grid):
    """Interleaved tiles are cut in the flattened list at multiples of 2048
    elements from each tensor's start (4 KB of a bf16 stream: measured, such
    cuts stream 1-2 % faster than 8K tiles cut per tensor and 18 % faster
    than cuts on 16-byte boundaries), except the cuts that end a tile of the
    last round, which fall on multiples of 256 so that every CTA's quota is
    the same to 256 elements: at most one such cut per CTA, and on a single
    tensor no CTA carries more than 256 elements beyond the mean.  Where the
    last rounds are left claimable instead (about 12 % of the rounds, in
    tiles claimed at run time), the CTAs' own shares agree to a cut unit."""
    entries = [_fake(i << 34, n, 1) for i, n in enumerate(sizes)]
    chunks = _check_partition(entries, 1, grid)
    load = np.zeros(grid, np.int64)
    claimable = 0
    off_grid = 0
    for c in chunks:
        if c.cta >= 0:
            load[c.cta] += c.len
        else:
            claimable += c.len
        assert c.offset % 256 == 0, "cut off the 256-element grid"
        off_grid += c.offset % 2048 != 0
    assert off_grid <= grid, (off_grid, grid)
    total = sum(sizes)
    # each CTA's own share (CTA 0 apart, 4096 elements short): the quota less
    # the last rounds, which are either dealt or left claimable
    own = (total - claimable - load[0]) / (grid - 1)
    rest = load[1:]
    if len(sizes) == 1:
        assert rest.max() - own <= (2048 if claimable else 256), (rest.max(), own)
        assert own - rest.min() <= (2048 if claimable else 512), (rest.min(), own)
        if claimable:
            # the relief may fall in the claimed rounds: CTA 0 then claims less
            assert load[0] <= own + 2048, (load[0], own)
        else:
            assert abs(own - load[0] - 4096) <= 512, (load[0], own)
    else:
        # each tensor's own cut grid moves a cut by up to 2047 elements
        assert rest.max() - own <= 2048 * len(sizes) + 2048, (rest.max(), own)
        assert own - load[0] >= 4096 - 2048 * len(sizes) - 512, (load[0], own)
    if total / grid >= 100 * 8192:
        assert load.max() <= 1.01 * total / grid, (load.max(), total / grid)
    if claimable and len(sizes) == 1:
        # claimable tiles shrink towards the end: the last claims are
        # single 2048-element cut units, the first are whole tiles
        tail = [c.len for c in chunks if c.cta < 0]
        assert max(tail[-grid:]) <= 2048 and tail[0] == 8192, (tail[:3], tail[-3:])
        # non-increasing (the very last may be cut short by the list's end)
        assert all(a >= b for a, b in zip(tail[:-2], tail[1:-1])), "claimable sizes grow"


def test_partition_misaligned_bases_take_head_or_element_path():
    # same skew on every stream: a short element-path head re-aligns them
    e_same = [_fake(0, 1000, 0, skew=(3, 3, 3, 3, 3))]
    ch = _check_partition(e_same, 0, 4)
    assert ch[0].vec == 0 and ch[0].len == 5 and all(c.vec for c in ch[1:])
    # different skews: no head works, whole tensor on the element path
    e_diff = [_fake(0, 1000, 0, skew=(1, 0, 0, 0, 0))]
    ch = _check_partition(e_diff, 0, 4)
    assert all(c.vec == 0 for c in ch)
    # mixed mode: fp32 streams 1 element (4 B) and bf16 streams 5 elements
    # (10 B) past a 16-B boundary: a 3-element head aligns all five
    e_mix = [_fake(0, 999, 1, skew=(1, 5, 1, 1, 5))]
    ch = _check_partition(e_mix, 1, 3)
    assert ch[0].vec == 0 and ch[0].len == 3 and all(c.vec for c in ch[1:])
    # remainder mode: bf16 param/remainder 5 elements and fp32 moments 1
    # element past a boundary: the same 3-element head aligns all five
    e_rem = [_fake(0, 999, 2, skew=(5, 5, 1, 1, 5))]
    ch = _check_partition(e_rem, 2, 3)
    assert ch[0].vec == 0 and ch[0].len == 3 and all(c.vec for c in ch[1:])
    # fp32 moments must be 4-byte aligned in remainder mode
    with pytest.raises(A.AdamWError) as e:
        A.adamw_plan_chunks([(16, 16, 34, 48, 64, 10)], 2, 2)
    assert e.value.status == A.ADAMW_ERR_MISALIGNED


@pytest.mark.parametrize("mode", A.ANYPREC_MODES)
def test_anyprec_partition_respects_each_stream_type(mode):
    """Every any-precision mode partitions like the others, with 16-byte
    aligned vector chunks under its own element sizes, whatever the skew of
    each base (a skew no head can fix sends the tensor down the element
    path)."""
    sizes = [1, 9, 4095, 65537, 0, 257, 1 << 20]
    for skew in ((0, 0, 0, 0, 0), (1, 0, 0, 0, 0), (0, 3, 1, 1, 1), (5, 5, 5, 5, 5)):
        es = ELEM_SIZES[mode]
        entries = [_fake(i << 30, n, mode, skew) for i, n in enumerate(sizes)]
        if es[4] == 0:
            entries = [e[:4] + (0,) + e[5:] for e in entries]
        for grid in (1, 7, 456):
            _check_partition(entries, mode, grid)


def test_anyprec_mode_validation():
    """Modes 16..27 are valid except 28..31 (fp32 compensation without Kahan
    summation); 5..15 and 32 are not modes; an fp32 buffer must be 4-byte
    aligned; without Kahan summation aux may be NULL."""
    for mode in list(range(5, 16)) + [28, 29, 30, 31, 32, -1]:
        with pytest.raises(A.AdamWError) as e:
            A.adamw_plan_chunks([_fake(0, 10, 0)], mode, 2)
        assert e.value.status == A.ADAMW_ERR_INVALID_ARG, mode
    assert len(A.ANYPREC_MODES) == 12
    for mode in A.ANYPREC_MODES:
        es = ELEM_SIZES[mode]
        ent = _fake(0, 10, mode)
        if es[4] == 0:
            ent = ent[:4] + (0,) + ent[5:]
        assert len(A.adamw_plan_chunks([ent], mode, 2)) >= 1
        for s in (2, 3, 4):
            if es[s] == 4:
                bad = list(ent)
                bad[s] += 2
                with pytest.raises(A.AdamWError) as e:
                    A.adamw_plan_chunks([tuple(bad)], mode, 2)
                assert e.value.status == A.ADAMW_ERR_MISALIGNED


def test_buffer_dtypes_follow_the_flags():
    import torch
    bf, f32 = torch.bfloat16, torch.float32
    assert A.buffer_dtypes(A.MODE_ANYPREC) == A.buffer_dtypes(A.MODE_BF16_KAHAN)
    assert A.buffer_dtypes(A.MODE_ANYPREC | A.ANYPREC_NO_KAHAN) == A.buffer_dtypes(A.MODE_BF16_PLAIN)
    assert A.buffer_dtypes(A.MODE_ANYPREC | A.ANYPREC_V_FP32) == A.buffer_dtypes(A.MODE_BF16_KAHAN_FP32_VAR)
    assert A.buffer_dtypes(A.MODE_ANYPREC | 7) == (bf, bf, f32, f32, f32)
    assert A.buffer_dtypes(A.MODE_ANYPREC | 9) == (bf, bf, f32, bf, None)
    with pytest.raises(ValueError):
        A.buffer_dtypes(A.MODE_ANYPREC | 12)


def test_opt_1_3b_partition():
    from adamw_optimizer_step_sm_gb300 import workloads as W
    w = W.WORKLOADS["opt1.3b_bf16_kahan"]
    offs, _ = W.tensor_offsets(w.numels)
    entries = [tuple(b + (k + 1) * (1 << 40) for k in range(5)) + (n,)
               for b, n in zip((2 * o for o in offs), w.numels)]
    ch = _check_partition(entries, 0, 152 * 3)
    assert all(c.vec for c in ch)


def test_validation_errors():
    with pytest.raises(A.AdamWError) as e:
        A.adamw_plan_chunks([_fake(0, 10, 0, skew=(0, 0, 0, 0, 0))[:4] + (1,) + (10,)], 0, 2)
    assert e.value.status == A.ADAMW_ERR_MISALIGNED
    with pytest.raises(A.AdamWError) as e:
        A.adamw_plan_chunks([(0, 0, 0, 0, 0, 10)], 0, 2)
    assert e.value.status == A.ADAMW_ERR_INVALID_ARG
    with pytest.raises(A.AdamWError) as e:
        A.adamw_plan_chunks([_fake(0, -1)], 0, 2)
    assert e.value.status == A.ADAMW_ERR_INVALID_ARG
    with pytest.raises(A.AdamWError) as e:
        A.adamw_plan_chunks([_fake(0, 10)], 7, 2)
    assert e.value.status == A.ADAMW_ERR_INVALID_ARG
    # fp32 master must be 4-byte aligned in mixed mode
    with pytest.raises(A.AdamWError) as e:
        A.adamw_plan_chunks([_fake(0, 10, 1, skew=(0, 0, 0, 0, 0))[:0] + (2, 16, 32, 64, 96, 10)], 1, 2)
    assert e.value.status == A.ADAMW_ERR_MISALIGNED
    # zero-length tensors may have NULL buffers
    assert A.adamw_plan_chunks([(0, 0, 0, 0, 0, 0)], 0, 2) == []


@pytest.mark.parametrize("bad", [dict(beta1=1.0), dict(beta2=-0.1), dict(eps=0.0),
                                 dict(lr=-1e-3), dict(weight_decay=-0.1),
                                 dict(lr=float("nan")), dict(max_grad_norm=float("inf"))])
def test_hparam_validation(bad):
    hp = A.hparams(**bad)
    with pytest.raises(A.AdamWError) as e:
        A.adamw_step_scalars(hp, 1)
    assert e.value.status == A.ADAMW_ERR_INVALID_ARG


def test_step_zero_rejected():
    with pytest.raises(A.AdamWError):
        A.adamw_step_scalars(A.hparams(), 0)


@pytest.mark.parametrize("t", [1, 2, 3, 10, 1000, 10**9])
@pytest.mark.parametrize("betas", [(0.9, 0.95), (0.9, 0.999), (0.0, 0.0), (0.5, 0.25)])
def test_step_scalars_agree_with_the_oracle(t, betas):
    """Library and oracle compute the per-step scalars independently from the
    same definition; they must agree bit for bit."""
    hp = A.hparams(lr=2e-4, beta1=betas[0], beta2=betas[1], weight_decay=0.1)
    ohp = oracle.hparams(lr=2e-4, beta1=betas[0], beta2=betas[1], weight_decay=0.1)
    ours = np.array(A.adamw_step_scalars(hp, t), np.float32)
    ref = oracle.load().step_scalars(ohp, t)
    assert np.array_equal(ours.view(np.uint32), ref.view(np.uint32))


def test_gpu_entry_points_fail_loudly_without_a_gpu():
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    with pytest.raises(A.AdamWError) as e:
        A.adamw_plan_create([_fake(0, 64)], 0)
    assert e.value.status == A.ADAMW_ERR_CUDA


@pytest.mark.parametrize("warmup,total", [(500, 1000), (0, 100), (1, 1), (7, 3), (500, 500), (3, 10**7)])
def test_lr_schedule_agrees_with_the_oracle(warmup, total):
    """The library's and the oracle's linear warm-up schedules, computed
    independently from the recipe's definition, agree bit for bit."""
    o = oracle.load()
    for t in list(range(1, 30)) + [warmup, warmup + 1, warmup + 2, total - 1, total, total + 1,
                                   total + 5, 10**6]:
        if t < 1:
            continue
        a = np.float32(A.adamw_lr_linear_warmup(np.float32(2e-4), t, warmup, total))
        b = np.float32(o.lr_linear_warmup(np.float32(2e-4), t, warmup, total))
        assert a.view(np.uint32) == b.view(np.uint32), (t, a, b)


def test_optimizer_options_map_to_storage_modes():
    import torch
    from adamw_optimizer_step_sm_gb300 import optim as OPT
    bf, f32 = torch.bfloat16, torch.float32
    assert OPT.storage_mode(True, bf, bf, bf) == A.MODE_ANYPREC
    assert OPT.storage_mode(True, f32, f32, f32) == A.MODE_ANYPREC | 7
    assert OPT.storage_mode(False, f32, bf, f32) == A.MODE_ANYPREC | 9   # c type unused
    assert all(OPT.storage_mode(k, m, v, c) in A.ANYPREC_MODES
               for k in (True, False) for m in (bf, f32) for v in (bf, f32) for c in (bf, f32))
    with pytest.raises(ValueError):
        OPT.storage_mode(True, torch.float16, bf, bf)
    with pytest.raises(ValueError):
        OPT.AnyPrecisionAdamW([torch.zeros(2, dtype=bf)], lr=-1.0)
    with pytest.raises(ValueError):
        OPT.AnyPrecisionAdamW([torch.zeros(2, dtype=bf)], betas=(0.9, 1.0))
    with pytest.raises(TypeError):   # parameters must be bf16 CUDA tensors
        OPT.AnyPrecisionAdamW([torch.zeros(2, dtype=bf)])


def test_partition_properties_on_random_lists():
    """200 random lists (1-60 tensors of 0 to 300,000 elements, a random
    storage mode, each stream's base skewed by a random number of elements,
    a random grid from 1 to 1216): every element lands in exactly one chunk,
    chunks come in CTA order, vector chunks start 16-byte aligned in every
    stream, and interleaved cuts inside a vector body fall on the
    2048-element grid from the body's start (256 for the one cut per CTA
    that ends its last tile)."""
    rng = np.random.default_rng(2024)
    modes = [0, 1, 2, 3, 4] + list(A.ANYPREC_MODES)
    for case in range(200):
        mode = int(rng.choice(modes))
        es = ELEM_SIZES[mode]
        n_t = int(rng.integers(1, 61))
        sizes = rng.integers(0, 300_001, n_t)
        sizes[rng.random(n_t) < 0.2] = rng.integers(0, 9, int(np.sum(rng.random(n_t) < 0.2)) or 1)[0]
        entries = []
        for k, n in enumerate(sizes):
            skew = [int(rng.integers(0, 8)) if rng.random() < 0.3 else 0 for _ in range(5)]
            base = (k + 1) << 36
            e = tuple(base + (s + 1) * (1 << 32) + sk * max(es[s], 1) for s, sk in enumerate(skew))
            if es[4] == 0:
                e = e[:4] + (0,)
            entries.append(e + (int(n),))
        grid = int(rng.integers(1, 1217))
        chunks = _check_partition(entries, mode, grid)
        # cuts inside a vector body: on the 2048-element grid of the body
        # (interleaved partition; the last round's tile ends on its
        # 256-element grid, at most one per CTA) or on whole vectors
        # (contiguous ranges)
        interleaved = int(sizes.sum()) >= 2 * grid * 8192
        step = 256 if interleaved else 8
        heads = {}
        for c in chunks:
            if c.vec:
                heads.setdefault(c.tensor, []).append(c.offset)
        coarse = 0
        for k, offs in heads.items():
            head = min(offs)
            assert all((o - head) % step == 0 for o in offs), (case, k, step, sorted(offs)[:5])
            coarse += sum((o - head) % 2048 != 0 for o in offs)
        if interleaved:
            assert coarse <= grid, (case, coarse, grid)


def test_master_weight_optimizer_validates_its_options():
    import torch
    from adamw_optimizer_step_sm_gb300 import optim as OPT
    bf = torch.bfloat16
    with pytest.raises(ValueError):
        OPT.MasterWeightAdamW([torch.zeros(2, dtype=bf)], master="fp16")
    with pytest.raises(ValueError):
        OPT.MasterWeightAdamW([torch.zeros(2, dtype=bf)], eps=0.0)
    with pytest.raises(TypeError):   # bf16 CUDA model parameters only
        OPT.MasterWeightAdamW([torch.zeros(2, dtype=torch.float32)])
