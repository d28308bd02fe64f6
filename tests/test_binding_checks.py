"""The Python binding's argument checks (no GPU): the library sees raw
pointers, so every tensor's dtype, shape, layout and device is checked before
a call, with ValueError rather than assert."""
import pytest

torch = pytest.importorskip("torch")

from speculative_decoding_verification_68_gb300 import check_batch, check_outputs  # noqa: E402

K, V = 3, 40
CPU = torch.device("cpu")


def batch(B=4, dtype=torch.bfloat16):
    return dict(target=torch.zeros((B, K + 1, V), dtype=dtype), draft=torch.zeros((B, K, V), dtype=dtype),
                tokens=torch.zeros((B, K), dtype=torch.int32), temperature=torch.ones(B),
                uniforms=torch.zeros((B, K + 1)))


def check(b, max_batch=8, **kw):
    return check_batch(K, V, torch.bfloat16, max_batch, CPU, b["target"], b["draft"], b["tokens"],
                       b["temperature"], b["uniforms"], **kw)


def test_valid_batch_returns_its_size():
    assert check(batch(4)) == 4
    assert check(batch(0)) == 0
    b = batch(2)
    assert check_batch(K, V, torch.bfloat16, 8, CPU, b["target"], b["draft"], None, b["temperature"], None,
                       need_tokens=False, need_uniforms=False) == 2


@pytest.mark.parametrize("mutate, what", [
    (lambda b: b.update(target=b["target"].float()), "dtype"),
    (lambda b: b.update(draft=torch.zeros((4, K, V + 1), dtype=torch.bfloat16)), "shape"),
    (lambda b: b.update(draft=torch.zeros((4, K + 1, V), dtype=torch.bfloat16)), "shape"),
    (lambda b: b.update(tokens=b["tokens"].long()), "dtype"),
    (lambda b: b.update(tokens=torch.zeros((K, 4), dtype=torch.int32).t()), "contiguous"),
    (lambda b: b.update(temperature=torch.ones(5)), "shape"),
    (lambda b: b.update(uniforms=torch.zeros((4, K))), "shape"),
    (lambda b: b.update(uniforms=None), "required"),
    (lambda b: b.update(target=torch.zeros((4, V), dtype=torch.bfloat16)), "target must be"),
])
def test_bad_inputs_raise(mutate, what):
    b = batch(4)
    mutate(b)
    with pytest.raises(ValueError, match=what):
        check(b)


def test_batch_above_capacity_raises():
    with pytest.raises(ValueError, match="max_batch"):
        check(batch(9), max_batch=8)


def test_device_mismatch_raises():
    b = batch(2)
    with pytest.raises(ValueError, match="expected cuda"):
        check_batch(K, V, torch.bfloat16, 8, torch.device("cuda", 0), b["target"], b["draft"], b["tokens"],
                    b["temperature"], b["uniforms"])


def test_outputs_checked():
    B = 3
    good = {"tokens": torch.zeros((B, K + 1), dtype=torch.int32), "tau": torch.zeros(B, dtype=torch.int32),
            "tv": torch.zeros((B, K))}
    check_outputs(good, B, K, V, torch.bfloat16, CPU)
    with pytest.raises(ValueError, match="required"):
        check_outputs({"tokens": good["tokens"]}, B, K, V, torch.bfloat16, CPU)
    with pytest.raises(ValueError, match="shape"):
        check_outputs(dict(good, tv=torch.zeros((B, K + 1))), B, K, V, torch.bfloat16, CPU)
    with pytest.raises(ValueError, match="unknown"):
        check_outputs(dict(good, extra=torch.zeros(1)), B, K, V, torch.bfloat16, CPU)
    grad = {"grad": torch.zeros((B, K, V), dtype=torch.float32)}
    with pytest.raises(ValueError, match="dtype"):
        check_outputs(grad, B, K, V, torch.bfloat16, CPU, required=("grad",))
