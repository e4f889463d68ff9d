"""Loading the seeded synthetic workloads (the `synth` module) into a decode context.

Weights are drawn as fp32 N(0, 0.02) on the host and handed to mie_load_weights as
fp32, so the GPU quantises them with its own kernels; norm gains stay at 1.
"""
from __future__ import annotations

from ._binding import FMT, Model


def config_for(shape, n_kv_blocks: int, max_pos: int, max_slots: int = 1, layers: int | None = None) -> dict:
    return dict(n_layers=shape.n_layers if layers is None else layers, d_model=shape.d_model,
                n_heads=shape.n_heads, n_kv_heads=shape.n_kv_heads, head_dim=shape.head_dim,
                ffn=shape.ffn, vocab=shape.vocab, tied=int(shape.tied), block_size=shape.block_size,
                act_bf16=int(shape.act_bf16), rms_eps=shape.rms_eps, rope_theta=shape.rope_theta,
                wfmt=FMT[shape.wfmt], head_fmt=FMT[shape.head_fmt], embed_fmt=FMT[shape.wfmt],
                n_kv_blocks=n_kv_blocks, max_slots=max_slots, max_pos=max_pos)


def build_gpu_model(shape, n_kv_blocks: int, max_pos: int, max_slots: int = 1, layers: int | None = None,
                    stream=None) -> Model:
    nl = shape.n_layers if layers is None else layers
    m = Model(config_for(shape, n_kv_blocks, max_pos, max_slots, nl), stream)
    for name, _, _ in shape.tensors():
        if name.startswith("l") and int(name[1:].split(".")[0]) >= nl:
            continue
        m.load_weights(name, shape.weight(name), "f32")
    return m


def prompt_tokens(shape, n: int, stream: int = 0):
    return shape.tokens(n, stream)
