"""Planted mistakes: each mutant of the oracle's C source must fail a pin.

A mutant is the oracle source with one plausible slip (a wrong index, a
dropped term, a flipped sign, a transposed operand).  It is compiled to a
temporary library on the CPU and the pin suite is run against it; the test
passes only if the pins reject every mutant.  Nothing here touches a GPU.
"""
import os
import subprocess
import sys

import pytest

from oracle.build import SRC

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

MUTANTS = {
    "gqa_head_interleaved": ("int h = kvh * G + g;", "int h = g * j->Hk + kvh;"),
    "gather_offset_shift": ("int off = i % bs;", "int off = (i + 1) % bs;"),
    "gather_block_off_by_one": ("int64_t phys = table[i / bs];", "int64_t phys = table[(i + 1) / bs];"),
    "cache_layout_transposed": ("int64_t row = ((phys * Hk + kvh) * bs + off) * (int64_t)D;",
                                "int64_t row = ((phys * bs + off) * Hk + kvh) * (int64_t)D;"),
    "scale_dropped": ("z[i] = scale * dot;", "z[i] = dot;"),
    "softmax_sign": ("double p = exp(z[i] - m);", "double p = exp(m - z[i]);"),
    "normaliser_dropped": ("        o[d] /= l;\n}", "        o[d] /= 1.0;\n}"),
    "merge_weight_drops_l": ("double w = lp[p] * exp(mp[p] - M);", "double w = exp(mp[p] - M);"),
    "blocks_floor_plus_one": ("return (n_tokens + block_size - 1) / block_size;",
                              "return n_tokens / block_size + 1;"),
    "f16_exponent_bias": ("v = ldexp((double)(m | 0x400), e - 25);", "v = ldexp((double)(m | 0x400), e - 24);"),
    "scatter_block_offset_swapped": ("size_t dst = (size_t)(((b * num_kv_heads + h) * block_size + o)) * row;",
                                     "size_t dst = (size_t)(((o * num_kv_heads + h) * block_size + b)) * row;"),
    "copy_direction_swapped": ("memcpy((char *)k_caches[l] + (size_t)dst * block_bytes,\n                   (const char *)k_caches[l] + (size_t)src * block_bytes",
                               "memcpy((char *)k_caches[l] + (size_t)src * block_bytes,\n                   (const char *)k_caches[l] + (size_t)dst * block_bytes"),
    "swap_direction_inverted": ("            if (direction == 0) {\n                memcpy(hk, gk, block_bytes);",
                                "            if (direction != 0) {\n                memcpy(hk, gk, block_bytes);"),
    "bf16_shift_15": ("uint32_t u = (uint32_t)b << 16;", "uint32_t u = (uint32_t)b << 15;"),
    "attend_drops_last_token": ("    for (int i = 0; i < L; ++i) {\n        double p = exp(z[i] - m);",
                                "    for (int i = 0; i < L - 1; ++i) {\n        double p = exp(z[i] - m);"),
    "partitions_overlap_by_one": ("int i0 = p * P, i1 = i0 + P < L ? i0 + P : L;",
                                  "int i0 = p * P, i1 = i0 + P + 1 < L ? i0 + P + 1 : L;"),
    "merge_exponent_flipped": ("double w = lp[p] * exp(mp[p] - M);", "double w = lp[p] * exp(M - mp[p]);"),
    "scatter_slot0_is_padding": ("        if (slot < 0)\n            continue;",
                                 "        if (slot <= 0)\n            continue;"),
    "swap_host_index_is_gpu_index": ("char *hk = (char *)host_k[l] + (size_t)h * block_bytes;",
                                     "char *hk = (char *)host_k[l] + (size_t)(g % host_blocks) * block_bytes;"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_reject_mutant(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation site for {name} not found exactly once"
    mutant_src = tmp_path / "mutant.c"
    mutant_src.write_text(src.replace(old, new))
    lib = tmp_path / "libmutant.so"
    subprocess.run(["gcc", "-std=c11", "-O1", "-fPIC", "-shared", "-D_POSIX_C_SOURCE=200809L",
                    str(mutant_src), "-o", str(lib), "-lm", "-lpthread"], check=True)
    env = dict(os.environ, PKV_ORACLE_LIB=str(lib))
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle_pins.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode != 0, f"mutant {name} passed every pin:\n{r.stdout[-2000:]}"


# Planted mistakes in the oracle's Python block manager (on-demand blocks,
# fork, copy-on-write, free, prefix caching): the mutated module is put in place of
# oracle.block_manager before the pin suite imports it.
BM_MUTANTS = {
    "cow_on_any_write": ("            if self.refcount[b] > 1:", "            if self.refcount[b] >= 1:"),
    "cow_keeps_old_reference": ("                self.refcount[b] -= 1\n                table[j] = nb",
                                "                table[j] = nb"),
    "fork_takes_no_reference": ("        for b in self.tables[child]:\n            self.refcount[b] += 1",
                                "        for b in self.tables[child]:\n            pass"),
    "free_never_returns_blocks": ("            if self.refcount[b] == 0:\n                self.free.append(b)",
                                  "            if self.refcount[b] < 0:\n                self.free.append(b)"),
    "blocks_rounded_down": ("    return -(-n_tokens // block_size)", "    return n_tokens // block_size"),
    # prefix caching
    "prefix_key_is_the_block_alone": ("        return toks[:(k + 1) * self.block_size]",
                                      "        return toks[k * self.block_size:(k + 1) * self.block_size]"),
    "reused_blocks_not_held": ("        for b in reused:\n            self._hold(b)",
                               "        for b in reused:\n            pass"),
    "evicts_latest_released": ("            b = self.idle.pop(0)", "            b = self.idle.pop()"),
    "cached_block_written_in_place": ("        if self.holders[b] == 1 and b not in self.key:",
                                      "        if self.holders[b] == 1:"),
    "refusal_counts_idle_reused_as_free": ("        if self.available() - idle_reused < fresh:",
                                           "        if self.available() < fresh:"),
    "second_commit_replaces_entry": ("            if b not in self.key and prefix not in self.entry:",
                                     "            if b not in self.key:"),
}


@pytest.mark.parametrize("name", sorted(BM_MUTANTS))
def test_pins_reject_block_manager_mutant(name, tmp_path):
    old, new = BM_MUTANTS[name]
    path = os.path.join(ROOT, "oracle", "block_manager.py")
    src = open(path).read()
    assert src.count(old) == 1, f"mutation site for {name} not found exactly once"
    mutant = tmp_path / "block_manager.py"
    mutant.write_text(src.replace(old, new))
    code = (
        "import importlib.util, sys\n"
        f"sys.path.insert(0, {ROOT!r})\n"
        "import oracle, pytest\n"
        f"spec = importlib.util.spec_from_file_location('oracle.block_manager', {str(mutant)!r})\n"
        "mod = importlib.util.module_from_spec(spec)\n"
        "spec.loader.exec_module(mod)\n"
        "sys.modules['oracle.block_manager'] = mod\n"
        "oracle.block_manager = mod\n"
        f"sys.exit(pytest.main(['-x', '-q', '-p', 'no:cacheprovider', "
        f"{os.path.join(ROOT, 'tests', 'test_oracle_pins.py')!r}]))\n")
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, capture_output=True, text=True,
                       timeout=600)
    assert r.returncode != 0, f"mutant {name} passed every pin:\n{r.stdout[-2000:]}"
    # a pin failed (status 1), not the import or collection (status 2 and up)
    assert r.returncode == 1, f"pytest status {r.returncode}:\n{r.stdout[-2000:]}{r.stderr[-2000:]}"
