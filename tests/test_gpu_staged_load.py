"""amk_load_weights_staged: the weights in host memory, each group of
matrices copied through a device staging buffer and repacked from there.
The packed model must be the one amk_load_weights builds from device
weights, so decode steps from both give bit-identical logits and K,V."""
import pytest
import torch

from workload import configs as wc
from workload import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import __graft_entry__
    __graft_entry__.build()
    d = torch.device("cuda:0")
    torch.cuda.set_device(d)
    return d


@pytest.fixture(scope="module")
def amk(dev):
    from decode_megakernel_gb300 import amk as m
    return m


def variant(name):
    base = dict(wc.TINY.__dict__)
    if name == "int8":
        base.update(weight_format="int8")
    elif name == "int4":
        base.update(weight_format="int4", ffn=768)
    elif name == "tied":
        base.update(tied_embeddings=True)
    return wc.ModelConfig(**base)


@pytest.mark.parametrize("name", ["tiny", "int8", "int4", "tied"])
def test_host_weights_load_the_same_model(amk, dev, name):
    cfg = variant(name)
    P, steps = 16, 6
    max_seq = P + steps
    w_dev = synth.model_weights(cfg, seed=21, device=dev)
    w_host = w_dev.to("cpu")
    a = amk.Decoder(w_dev, max_seq)
    b = amk.Decoder(w_host, max_seq, device=dev)
    del w_dev
    torch.cuda.empty_cache()
    prompt = synth.prompt_tokens(cfg, P).tolist()
    a.prefill(prompt, 0)
    b.prefill(prompt, 0)
    la = torch.empty(cfg.vocab, dtype=torch.float32, device=dev)
    lb = torch.empty_like(la)
    for i, t in enumerate(synth.decode_tokens(cfg, steps).tolist()):
        a.decode_step(t, P + i, la)
        b.decode_step(t, P + i, lb)
        a.sync()
        b.sync()
        assert torch.equal(la, lb), (name, i)
    assert torch.equal(a.kv, b.kv)
    a.close()
    b.close()


def test_full_size_host_load_matches(amk, dev):
    """The 1B model (2.5 GB) loaded from host memory through a 67 MB
    staging buffer decodes exactly as the device-loaded one."""
    wl = wc.workload("llama1b")
    cfg = wl.model
    assert amk.amk_weights_staging_bytes(amk.make_config(cfg, 64)) < 100 << 20
    w_dev = synth.model_weights(cfg, seed=synth.WEIGHT_SEED, device=dev)
    a = amk.Decoder(w_dev, 64)
    w_host = w_dev.to("cpu")
    b = amk.Decoder(w_host, 64, device=dev)
    del w_dev
    torch.cuda.empty_cache()
    la = torch.empty(cfg.vocab, dtype=torch.float32, device=dev)
    lb = torch.empty_like(la)
    for i, t in enumerate(synth.decode_tokens(cfg, 4).tolist()):
        a.decode_step(t, i, la)
        b.decode_step(t, i, lb)
        a.sync()
        b.sync()
        assert torch.equal(la, lb), i
    a.close()
    b.close()
