"""pa_slot_mapping_and_cache (and its FP8 form) against pa_slot_mapping
followed by pa_reshape_and_cache: the same slots, the same error flags and
bit-identical pools, including tokens outside the batch or the table, table
entries outside the pool (slot -1, nothing written) and padding tokens."""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def B():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_cache_96_gb300 import binding
    return binding


def _case(seed, fp8):
    rng = np.random.default_rng(seed)
    S, MB, N, bs, Hkv, d, T = 6, 8, 64, 16, 2, 128, 57
    tables = rng.permutation(N)[: S * MB].reshape(S, MB).astype(np.int32)
    tables[2, 3] = N + 5          # an entry outside the pool
    tables[4, 1] = -2
    # distinct (sequence, position) pairs: two tokens on one slot would race
    flat = rng.choice(S * MB * bs, size=T, replace=False)
    seq = (flat // (MB * bs)).astype(np.int32)
    pos = (flat % (MB * bs)).astype(np.int32)
    seq[5], pos[6], pos[7] = S + 1, -3, MB * bs   # outside the batch / the table
    seq[8], pos[8] = 2, 3 * bs + 4                 # lands on the bad entry
    key = torch.randn(T, Hkv, d, dtype=torch.bfloat16, device="cuda")
    val = torch.randn(T, Hkv, d, dtype=torch.bfloat16, device="cuda")
    if fp8:
        kc = torch.full((N, bs, Hkv, d), 0x7F, dtype=torch.uint8, device="cuda")
    else:
        kc = torch.full((N, bs, Hkv, d), 0x7FC0, dtype=torch.int16,
                        device="cuda").view(torch.bfloat16)
    return (torch.from_numpy(tables).cuda(), torch.from_numpy(seq).cuda(),
            torch.from_numpy(pos).cuda(), key, val, kc, kc.clone())


@pytest.mark.parametrize("fp8", [False, True])
def test_fused_matches_two_calls(B, fp8):
    tables, seq, pos, key, val, kc, vc = _case(5, fp8)
    T = seq.shape[0]
    N = kc.shape[0]
    kc2, vc2 = kc.clone(), vc.clone()
    slots_a = torch.full((T,), 123, dtype=torch.int32, device="cuda")
    slots_b = slots_a.clone()
    err_a = torch.zeros(1, dtype=torch.int32, device="cuda")
    err_b = torch.zeros(1, dtype=torch.int32, device="cuda")
    B.pa_slot_mapping(slots_a, tables, seq, pos, kc.shape[1], N, error_word=err_a)
    if fp8:
        B.pa_reshape_and_cache_fp8(key, val, kc, vc, slots_a, 0.02, 0.03, error_word=err_a)
    else:
        B.pa_reshape_and_cache(key, val, kc, vc, slots_a, error_word=err_a)
    B.pa_slot_mapping_and_cache(slots_b, tables, seq, pos, key, val, kc2, vc2, 0.02, 0.03,
                                error_word=err_b)
    torch.cuda.synchronize()
    assert torch.equal(slots_a, slots_b)
    assert int(err_a.item()) == int(err_b.item()) != 0
    sa = slots_a.cpu().numpy()
    assert (sa[[5, 6, 7, 8]] == -1).all()
    bits = (lambda t: t.view(torch.uint8)) if fp8 else (lambda t: t.view(torch.int16))
    assert torch.equal(bits(kc), bits(kc2))
    assert torch.equal(bits(vc), bits(vc2))
