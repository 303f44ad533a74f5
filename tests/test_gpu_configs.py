"""The five workload presets at full size on the GPU, in the launch
configuration the benchmark times: sampled sequences checked against the
oracle step by step (scatter, copy-on-write copies and attention)."""
import numpy as np
import pytest
import torch

from tests.gpu_support import TOL, SampledOracle, max_err
from workloads import CONFIGS, PagedDecodeWorkload
from workloads.runner import DeviceState

pytestmark = pytest.mark.gpu

SEED_BASE = 311 * 100


def run_config(cfg, seed, steps, samples, partition_size=None, pool_blocks=None):
    w = PagedDecodeWorkload(cfg, seed, total_steps=max(steps, 1), pool_blocks=pool_blocks)
    state = DeviceState(cfg, w, seed)
    inputs = [w.next_step() for _ in range(steps)]
    rng = np.random.default_rng(seed)
    seqs = sorted(rng.choice(w.num_seqs, size=min(samples, w.num_seqs), replace=False).tolist())
    orc = SampledOracle(state, seqs, inputs)       # snapshot before any library kernel runs
    worst = 0.0
    for inp in inputs:
        ds = state.to_device(inp, value_device="cpu")   # same values for both sides
        state.run_step(ds, partition_size=partition_size)
        torch.cuda.synchronize()
        assert state.status.item() == 0
        orc.apply_step(inp, ds.key.cpu(), ds.value.cpu())
        ref = orc.attention(inp, ds.q.cpu())
        got = state.out[seqs].to(torch.float64).cpu().numpy()
        err = max_err(got, ref)
        worst = max(worst, err)
        assert err <= TOL[cfg.dtype], f"{cfg.name} step {inp.step}: max err {err}"
    return worst


def test_tiny_f32_every_sequence():
    cfg = CONFIGS[0]
    run_config(cfg, SEED_BASE + 0, steps=cfg.steps, samples=cfg.num_seqs)


@pytest.mark.parametrize("idx", [1, 2, 3, 5])
def test_preset_sampled(idx):
    cfg = CONFIGS[idx]
    run_config(cfg, SEED_BASE + idx, steps=3, samples=6)


@pytest.mark.parametrize("bs", [8, 16, 32])
def test_long_context_sampled(bs):
    cfg = CONFIGS[4].with_(block_size=bs)
    free = torch.cuda.mem_get_info()[0]
    pool_bytes = min(cfg.pool_value, 0.8 * free)
    nb = int(pool_bytes // (2 * cfg.block_bytes))
    run_config(cfg, SEED_BASE + 4, steps=2, samples=2, pool_blocks=nb)


@pytest.mark.parametrize("idx", [3, 5])
def test_shared_presets_sampled_on_tcgen05(idx):
    """The two shared-prefix presets at full size on the tcgen05 kernel."""
    import paged_kv_cache_311_gb300 as pkv
    pkv.set_decode_engine("tcgen05")
    try:
        run_config(CONFIGS[idx], SEED_BASE + idx, steps=3, samples=6)
        assert pkv.last_decode_engine() == "tcgen05"
    finally:
        pkv.set_decode_engine("auto")


@pytest.mark.parametrize("idx", [1, 2])
def test_full_step_in_the_cache_dtype_every_sequence(idx):
    """One full-size step of the Llama-7B (fp16) and Llama-13B (bf16)
    workloads with the output in the cache's dtype, as the benchmark runs it,
    checked on every sequence: the 16-bit output is the fp32 result of the
    same step rounded to nearest even (bit for bit), the fp32 result is within
    the attention tolerance of the oracle, and so the 16-bit output lies
    within one unit in the last place of the oracle's value rounded to that
    dtype, plus the fp32 result's own error."""
    import paged_kv_cache_311_gb300 as pkv
    from tests.gpu_support import ulp_bound
    from tests.util import DT
    cfg = CONFIGS[idx]
    seed = SEED_BASE + idx
    tdt = DT[cfg.dtype]
    w = PagedDecodeWorkload(cfg, seed, total_steps=1)
    state = DeviceState(cfg, w, seed, out_dtype=tdt)
    inp = w.next_step()
    orc = SampledOracle(state, list(range(w.num_seqs)), [inp])   # before any library kernel
    ds = state.to_device(inp, value_device="cpu")
    state.run_step(ds)                   # copy-on-write, scatter, decode into the 16-bit output
    out32 = torch.empty(state.out.shape, dtype=torch.float32, device=state.out.device)
    pkv.paged_attention_decode(out32, ds.q, state.k_cache, state.v_cache, ds.block_tables,
                               ds.context_lens, cfg.softmax_scale,
                               max_context_len=ds.max_context_len,
                               partition_size=cfg.partition_size, workspace=state.workspace,
                               device_status=state.status)
    torch.cuda.synchronize()
    assert state.status.item() == 0
    orc.apply_step(inp, ds.key.cpu(), ds.value.cpu())
    ref = orc.attention(inp, ds.q.cpu())
    got16 = state.out.double().cpu().numpy()
    got32 = out32.double().cpu().numpy()
    assert max_err(got32, ref) <= TOL[cfg.dtype]
    np.testing.assert_array_equal(got16, out32.to(tdt).double().cpu().numpy())
    rne = torch.from_numpy(ref).to(tdt).double().numpy()
    assert np.all(np.abs(got16 - rne) <= ulp_bound(ref, tdt) + np.abs(got32 - ref))
