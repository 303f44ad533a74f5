"""GPU parity of paged_attention_decode_shared (the shared-prefix path)
against the CPU oracle, which knows nothing about sharing: it just follows
every sequence's block table.

Cases mix groups of sequences forked from one prompt (their tables start with
the same block ids; the partially filled last prompt block is copied for all
but one member, as copy-on-write does), singleton sequences, groups larger
than one CTA can take (the planner cuts them), prefixes that are not a
multiple of the alignment, empty contexts and bad block ids."""
import numpy as np
import pytest
import torch

from tests.gpu_support import TOL, max_err
from tests.util import DT, raw_np

import oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True, params=["auto", "tcgen05"])
def shared_engine(request):
    """Every case on both shared-prefix kernels: "auto" takes the warp-level
    MMA kernel, "tcgen05" the tcgen05 kernel at head_dim 128 (head_dim 64 has
    none: PKV_EUNSUPPORTED)."""
    import paged_kv_cache_311_gb300 as pkv
    pkv.set_decode_engine(request.param)
    _ENGINE_NOW[0] = pkv.ENGINES[request.param]
    yield request.param
    pkv.set_decode_engine("auto")
    _ENGINE_NOW[0] = 0


def shared_case(seed, *, dtype="bf16", H=8, Hk=2, D=128, bs=16, groups=((300, (5, 40, 1, 70)),)):
    """groups: (prompt length, tail lengths of its members); a member with
    tail -1 is a singleton sequence of the given prompt length (no sharing)."""
    rng = np.random.default_rng(seed)
    seqs = []   # (logical K, V [L, Hk, D], table builder info)
    tables, lens = [], []
    next_block = [0]

    def take(n):
        b = list(range(next_block[0], next_block[0] + n))
        next_block[0] += n
        return b

    plan = []
    for prompt, tails in groups:
        full, rem = divmod(prompt, bs)
        shared_blocks = take(full + (1 if rem else 0))
        for i, t in enumerate(tails):
            if t < 0:
                plan.append(("single", prompt, None, None))
                continue
            plan.append(("member", prompt, t, (shared_blocks, full, rem, i == len(tails) - 1)))
    # assign blocks
    for kind, prompt, t, info in plan:
        if kind == "single":
            L = prompt
            tables.append(take(-(-L // bs)))
        else:
            shared_blocks, full, rem, keeps_partial = info
            L = prompt + t
            tb = list(shared_blocks[:full])
            if rem:
                tb.append(shared_blocks[full] if keeps_partial else take(1)[0])
            need = -(-L // bs) - len(tb)
            tb += take(max(need, 0))
            tables.append(tb[: -(-L // bs)] if L else [])
        lens.append(L)
    NB = next_block[0] + 2
    g = torch.Generator().manual_seed(seed)
    kc = torch.randn(NB, Hk, bs, D, generator=g).to(DT[dtype])
    vc = torch.randn(NB, Hk, bs, D, generator=g).to(DT[dtype])
    # copy-on-write copies hold the prompt's rows of the shared partial block
    for (kind, prompt, t, info), tb in zip(plan, tables):
        if kind == "member":
            shared_blocks, full, rem, keeps_partial = info
            if rem and not keeps_partial and len(tb) > full:
                kc[tb[full], :, :rem] = kc[shared_blocks[full], :, :rem]
                vc[tb[full], :, :rem] = vc[shared_blocks[full], :, :rem]
    MB = max(max(len(t) for t in tables), 1)
    bt = np.full((len(tables), MB), -1, dtype=np.int32)
    for i, t in enumerate(tables):
        bt[i, :len(t)] = t
    q = torch.randn(len(tables), H, D, generator=g).to(DT[dtype])
    return dict(q=q, k_cache=kc, v_cache=vc, block_tables=bt,
                context_lens=np.array(lens, dtype=np.int32), dtype=dtype, bs=bs, Hk=Hk,
                scale=float(np.float32(1.0 / np.sqrt(D))))


def run_shared(case, P=0, out_dtype=torch.float32, tables=None, plan_tables=None, calls=1,
               plan_lens=None):
    """Plans on the host from plan_tables and plan_lens (default: the tables
    and lengths given to the device), then runs the shared-prefix decode
    `calls` times with the same device plan; returns the last output and the
    OR of the status words."""
    import paged_kv_cache_311_gb300 as pkv
    dev = "cuda"
    q, kc, vc = case["q"].to(dev), case["k_cache"].to(dev), case["v_cache"].to(dev)
    dev_tables = case["block_tables"] if tables is None else tables
    bt = torch.as_tensor(dev_tables).to(dev)
    cl = torch.as_tensor(case["context_lens"]).to(dev)
    B, H, D = q.shape
    mcl = int(max(case["context_lens"].max(), 1))
    plan = pkv.plan_shared_prefix(dev_tables if plan_tables is None else plan_tables,
                                  case["context_lens"] if plan_lens is None else plan_lens,
                                  H, case["Hk"], D, case["bs"], mcl, P)
    plan_dev = plan.to(dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    out = None
    for _ in range(calls):
        out = torch.full(q.shape, float("nan"), dtype=out_dtype, device=dev)
        pkv.paged_attention_decode_shared(out, q, kc, vc, bt, cl, case["scale"], plan, plan_dev,
                                          max_context_len=mcl, device_status=st)
        torch.cuda.synchronize()
        assert pkv.last_decode_launches() == 2
        engine = int(pkv.load_library().pkv_last_decode_engine())
        if case["dtype"] != "f32":
            assert engine == (3 if _engine_now() == 3 else 2)
    # the device only reads the plan
    np.testing.assert_array_equal(plan_dev.cpu().numpy(), plan.host)
    return out.double().cpu().numpy(), int(st.item())


_ENGINE_NOW = [0]   # the engine code the fixture set


def _engine_now():
    return _ENGINE_NOW[0]


def oracle_out(case, tables=None):
    return oracle.paged_attention(raw_np(case["q"]), raw_np(case["k_cache"]), raw_np(case["v_cache"]),
                                  case["dtype"],
                                  case["block_tables"] if tables is None else tables,
                                  case["context_lens"], case["Hk"], case["scale"])


GROUPS = [
    (300, (5, 40, 1, 70)),          # partial last prompt block, 4 members
    (512, (0, 3, 17)),              # block-aligned prompt, a member with no tail
    (40, (100, -1, 9)),             # short prompt; a singleton in the middle
    (1000, (1, 2, 3, 4, 5, 6, 7)),  # more members than one CTA takes at G = 4
]


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("G", [1, 2, 4, 8])
@pytest.mark.parametrize("bs", [8, 16, 32])
def test_shared_prefix_matches_oracle(dtype, G, bs):
    case = shared_case(10 * G + bs, dtype=dtype, H=2 * G, Hk=2, D=128, bs=bs, groups=GROUPS)
    ref, st = oracle_out(case)
    assert st == 0
    for P in (0, 64, 512):
        got, gst = run_shared(case, P=P)
        assert gst == 0
        err = max_err(got, ref)
        assert err <= TOL[dtype], f"P={P} max err {err}"


def test_same_device_plan_serves_repeated_calls():
    case = shared_case(11, dtype="bf16", H=16, Hk=4, D=128, bs=16, groups=GROUPS)
    once, _ = run_shared(case, calls=1)
    thrice, st = run_shared(case, calls=3)
    assert st == 0
    np.testing.assert_array_equal(once, thrice)


def test_group_whose_tables_disagree_is_rejected_on_the_device():
    """The plan says the first group shares its prompt, but on the device one
    member's table points elsewhere in the shared part: that group's rows are
    zeroed and PKV_DEV_BAD_BLOCK is raised; the other groups are unaffected."""
    import paged_kv_cache_311_gb300 as pkv
    case = shared_case(12, dtype="bf16", H=8, Hk=2, D=128, bs=16, groups=GROUPS[:2])
    t = case["block_tables"].copy()
    t[2, 0] = case["k_cache"].shape[0] - 1          # member 2 of group 0, first prompt block
    got, st = run_shared(case, tables=t, plan_tables=case["block_tables"])
    assert st & pkv.DEV_BAD_BLOCK
    assert not got[:4].any()
    ref, _ = oracle_out(case)
    assert max_err(got[4:], ref[4:]) <= TOL["bf16"]


def test_plan_made_for_other_lengths_is_rejected_on_the_device():
    """The device holds one token fewer for sequence 1 than the plan was made
    for: its rows are zeroed and PKV_DEV_BAD_CONTEXT_LEN is raised; every
    other sequence is unaffected."""
    import paged_kv_cache_311_gb300 as pkv
    case = shared_case(13, dtype="bf16", H=8, Hk=2, D=128, bs=16, groups=GROUPS[:2])
    planned = case["context_lens"].copy()
    lens = planned.copy()
    lens[1] -= 1
    dev = dict(case, context_lens=lens)
    got, st = run_shared(dev, plan_lens=planned)
    assert st & pkv.DEV_BAD_CONTEXT_LEN
    assert not st & pkv.DEV_BAD_BLOCK
    assert not got[1].any()
    ref, _ = oracle_out(dev)
    keep = [i for i in range(len(lens)) if i != 1]
    assert max_err(got[keep], ref[keep]) <= TOL["bf16"]


@pytest.mark.parametrize("D", [64, 128])
def test_shared_prefix_half_output(D, shared_engine):
    """bf16 output is the fp32 result rounded to nearest even (bit-exact
    against the same plan with fp32 output), so it lies within one bf16 ulp
    of the oracle rounded to bf16, plus the fp32 result's own error; also
    for the plan cut into many 64-token items (one kv head fills the GPU).
    The tcgen05 kernel takes head_dim 128 only."""
    import paged_kv_cache_311_gb300 as pkv
    case = shared_case(3, dtype="bf16", H=8, Hk=1, D=D, bs=16, groups=GROUPS[:2])
    if D == 64 and shared_engine == "tcgen05":
        with pytest.raises(pkv.PkvError) as e:
            run_shared(case)
        assert e.value.status == -2
        return
    ref, _ = oracle_out(case)
    from tests.gpu_support import ulp_bound
    rne = torch.from_numpy(ref).to(torch.bfloat16).double().numpy()
    for P in (0, 512):
        got, st = run_shared(case, P=P, out_dtype=torch.bfloat16)
        got32, st32 = run_shared(case, P=P)
        assert st == 0 and st32 == 0
        np.testing.assert_array_equal(got, torch.from_numpy(got32).to(torch.bfloat16).double().numpy())
        assert max_err(got32, ref) <= TOL["bf16"]
        assert np.all(np.abs(got - rne) <= ulp_bound(ref, torch.bfloat16) + np.abs(got32 - ref)), f"P={P}"


def test_shared_prefix_equals_per_sequence_path():
    from tests.gpu_support import gpu_decode
    case = shared_case(5, dtype="bf16", H=16, Hk=4, D=128, bs=16, groups=GROUPS)
    a, _ = run_shared(case)
    b, _, _ = gpu_decode(case)
    assert max_err(a, b) <= 1e-5


def test_no_sharing_batch():
    case = shared_case(6, dtype="f16", H=8, Hk=8, D=128, bs=16,
                       groups=((100, (-1,)), (700, (-1,)), (33, (-1,))))
    ref, _ = oracle_out(case)
    got, st = run_shared(case)
    assert st == 0 and max_err(got, ref) <= TOL["f16"]


def test_empty_context_and_bad_block():
    import paged_kv_cache_311_gb300 as pkv
    case = shared_case(7, dtype="bf16", H=8, Hk=2, D=128, bs=16, groups=GROUPS[:1])
    lens = case["context_lens"].copy()
    lens[1] = 0
    c0 = dict(case, context_lens=lens)
    ref, _ = oracle_out(c0)
    got, st = run_shared(c0)
    assert st == 0 and not got[1].any() and max_err(got, ref) <= TOL["bf16"]
    t = case["block_tables"].copy()
    t[3, -1] = case["k_cache"].shape[0] + 3      # last member's own tail block
    got, st = run_shared(case, tables=t)
    assert st & pkv.DEV_BAD_BLOCK
    assert not got[3].any()
    ref, _ = oracle_out(case)
    assert max_err(got[:3], ref[:3]) <= TOL["bf16"]


def test_fp32_is_rejected():
    import paged_kv_cache_311_gb300 as pkv
    case = shared_case(8, dtype="f32", H=4, Hk=4, D=64, bs=16, groups=GROUPS[:1])
    with pytest.raises(pkv.PkvError) as e:
        run_shared(case)
    assert e.value.status == -2


def test_sharers_scattered_through_the_batch():
    """The batch order is shuffled, so each group's members are scattered
    (requests reusing a cached prompt arrive in any order): the planner still
    groups them and every output matches the oracle."""
    case = shared_case(14, dtype="bf16", H=16, Hk=4, D=128, bs=16, groups=GROUPS)
    perm = np.random.default_rng(14).permutation(len(case["context_lens"]))
    shuffled = dict(case, q=case["q"][torch.from_numpy(perm)],
                    block_tables=np.ascontiguousarray(case["block_tables"][perm]),
                    context_lens=np.ascontiguousarray(case["context_lens"][perm]))
    import paged_kv_cache_311_gb300 as pkv
    plan = pkv.plan_shared_prefix(shuffled["block_tables"], shuffled["context_lens"], 16, 4, 128, 16)
    h, B = plan.host, len(perm)
    base, iints = 8 + 2 * B, int(h[4])
    nrows = [int(h[base + i * iints + 1]) for i in range(plan.num_items)]
    assert max(nrows) > 4                    # groups formed: an item serves several sequences
    ref, _ = oracle_out(shuffled)
    for P in (0, 64):
        got, st = run_shared(shuffled, P=P)
        assert st == 0
        assert max_err(got, ref) <= TOL["bf16"], f"P={P}"


def growing_scores_case(seed, dtype="bf16", bs=16):
    """Keys carry a component along a fixed direction proportional to their
    logical position, and every query has that direction: scores climb by
    about 12 (log2 units) every 16 tokens, more than the kernels' 2^8 slack
    on a row's reference maximum, so every tile moves the running maxima and
    rescales the accumulators (on the tcgen05 kernel, O in tensor memory)."""
    case = shared_case(seed, dtype=dtype, H=8, Hk=2, D=128, bs=bs, groups=GROUPS)
    bt, lens = case["block_tables"], case["context_lens"]
    pos = {}
    for s in range(len(lens)):
        for j in range(-(-int(lens[s]) // bs)):
            for o in range(bs):
                pos[(int(bt[s, j]), o)] = j * bs + o   # shared blocks sit at the same position
    u = torch.zeros(128)
    u[:8] = 1.0
    kc = case["k_cache"].float()
    for (b, o), t in pos.items():
        kc[b, :, o, :] += 0.75 * t * u
    q = case["q"].float() + u
    return dict(case, k_cache=kc.to(DT[dtype]), q=q.to(DT[dtype]))


@pytest.mark.parametrize("bs", [8, 32])
def test_growing_scores_rescale_every_tile(bs, shared_engine):
    from tests.gpu_support import gpu_decode
    case = growing_scores_case(31 + bs, bs=bs)
    ref, st = oracle_out(case)
    assert st == 0
    for P in (0, 64):
        got, gst = run_shared(case, P=P)
        assert gst == 0
        assert max_err(got, ref) <= TOL["bf16"], f"shared P={P}"
    per_seq, pst, _ = gpu_decode(case)     # the per-sequence kernel's rescale too
    assert pst == 0 and max_err(per_seq, ref) <= TOL["bf16"]
